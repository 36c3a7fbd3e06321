"""CPU oracle of the decoder token step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. It compiles ``oracle.c`` with the host C compiler (no fast-math) and calls it through
ctypes. It shares no code with the CUDA library. See ``oracle.c`` for what is computed and the
passages each part follows.

Parity status of each part (what pins it, in ``tests/test_oracle_pins.py``):
dequantisation, rms_norm, norm_heads, rope, attention, the activations, matmul and the whole
forward are pinned against closed forms, invariants, library routines and brute force; absolute
logits of a random model beyond those pins are not given by the pages (no published outputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Iterable, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc -O2 -fopenmp, strict IEEE)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I64, I, D, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
        S = ctypes.c_char_p
        L.orc_create.restype = P
        L.orc_create.argtypes = [S, S, S, I64, ctypes.c_char_p, I]
        L.orc_last_error.restype = S
        L.orc_last_error.argtypes = [P]
        L.orc_add_tensor.restype = I
        L.orc_add_tensor.argtypes = [P, S, I, P, I, P, ctypes.c_size_t]
        L.orc_reset_kv.argtypes = [P]
        L.orc_write_kv.restype = I
        L.orc_write_kv.argtypes = [P, I, I64, I64, P, P]
        L.orc_read_kv.restype = I
        L.orc_read_kv.argtypes = [P, I, I64, I64, P, P]
        L.orc_set_kv_len.argtypes = [P, I64]
        L.orc_forward.restype = I
        L.orc_forward.argtypes = [P, P, I, I64, P, P, P]
        L.orc_steps.restype = I
        L.orc_steps.argtypes = [P, I]
        for f in ("orc_head_dim", "orc_rope_adjacent", "orc_window_pattern"):
            getattr(L, f).restype = I
            getattr(L, f).argtypes = [P]
        L.orc_destroy.argtypes = [P]
        L.orc_dequant.argtypes = [I, P, I64, P]
        L.orc_half_to_float.restype = F
        L.orc_half_to_float.argtypes = [ctypes.c_uint16]
        L.orc_round_to_half.restype = F
        L.orc_round_to_half.argtypes = [F]
        L.orc_set_kv_f16.restype = I
        L.orc_set_kv_f16.argtypes = [P, I]
        L.orc_rms_norm.argtypes = [P, P, I, D, P]
        L.orc_rope.argtypes = [P, I, I, I64, D, I]
        L.orc_attend.argtypes = [P, P, P, I, I64, I64, P]
        L.orc_act.argtypes = [I, P, I64, P]
        L.orc_matvec.argtypes = [I, P, I64, I64, P, P]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class OracleError(RuntimeError):
    pass


class Model:
    """An oracle decoder: archdef text + GGUF metadata + tensors (borrowed, kept alive here)."""

    def __init__(self, arch: str, archdef_text: str, metadata: Dict[str, str], max_ctx: int):
        L = lib()
        err = ctypes.create_string_buffer(512)
        md = "".join(f"{k}={v}\n" for k, v in metadata.items())
        h = L.orc_create(arch.encode(), archdef_text.encode(), md.encode(), max_ctx, err, 512)
        if not h:
            raise OracleError(err.value.decode())
        self._h = h
        self._keep = []
        self.n_embd = int(metadata[f"{metadata['general.architecture']}.embedding_length"])
        self.max_ctx = max_ctx
        self.n_vocab: Optional[int] = None

    def _check(self, rc: int) -> None:
        if rc != 0:
            raise OracleError(lib().orc_last_error(self._h).decode())

    def add_tensor(self, name: str, dtype: int, ne: Iterable[int], data: np.ndarray) -> None:
        ne = np.asarray(list(ne), dtype=np.int64)
        data = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
        self._keep += [ne, data]
        self._check(lib().orc_add_tensor(self._h, name.encode(), dtype, _ptr(ne), len(ne), _ptr(data),
                                         data.nbytes))
        if name == "token_embd.weight" and self.n_vocab is None:
            self.n_vocab = int(ne[1])
        if name == "output.weight":
            self.n_vocab = int(ne[1])

    def add_tensors(self, tensors) -> None:
        for t in tensors.values() if isinstance(tensors, dict) else tensors:
            self.add_tensor(t.name, t.dtype, t.ne, t.data)

    def steps(self, section: int) -> int:
        return lib().orc_steps(self._h, section)

    def reset_kv(self) -> None:
        lib().orc_reset_kv(self._h)

    def write_kv(self, layer: int, pos0: int, k: np.ndarray, v: np.ndarray) -> None:
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        self._check(lib().orc_write_kv(self._h, layer, pos0, k.shape[1], _ptr(k), _ptr(v)))

    def read_kv(self, layer: int, pos0: int, n: int, n_head_kv: int, head_dim: int):
        k = np.empty((n_head_kv, n, head_dim), np.float32)
        v = np.empty_like(k)
        self._check(lib().orc_read_kv(self._h, layer, pos0, n, _ptr(k), _ptr(v)))
        return k, v

    def set_kv_f16(self, on: bool = True) -> None:
        """Store keys and values rounded to f16 (the f16-KV configuration); before any forward."""
        self._check(lib().orc_set_kv_f16(self._h, int(on)))

    def set_kv_len(self, n: int) -> None:
        self._check(lib().orc_set_kv_len(self._h, n))

    def forward(self, tokens, pos: int, want_x: bool = False, n_layer: int = 0):
        """Logits of the last row (and optionally x after the epilogue / after each layer)."""
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
        logits = np.empty(self.n_vocab, np.float32)
        x = np.empty(self.n_embd, np.float32) if want_x else None
        lx = np.empty((n_layer, self.n_embd), np.float32) if n_layer else None
        self._check(lib().orc_forward(self._h, _ptr(t), len(t), pos, _ptr(logits),
                                      _ptr(x) if x is not None else None,
                                      _ptr(lx) if lx is not None else None))
        if want_x or n_layer:
            return logits, x, lx
        return logits

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().orc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def load_archdef(arch: str) -> str:
    """Read a shipped archdef text (input data, shared by both sides like the weights)."""
    root = os.path.dirname(_HERE)
    with open(os.path.join(root, "decoder_token_step_gb300", "archdefs", arch + ".archdef")) as f:
        return f.read()


def model_from_synth(cfg, tensors, max_ctx: int, archdef_text: Optional[str] = None) -> Model:
    import synth
    m = Model(cfg.arch, archdef_text or load_archdef(cfg.arch), synth.metadata(cfg, max_ctx), max_ctx)
    m.add_tensors(tensors)
    return m


# ---- single ops (pins) ----------------------------------------------------------------------

def dequant(dtype: int, row: np.ndarray, k: int) -> np.ndarray:
    row = np.ascontiguousarray(row).view(np.uint8)
    out = np.empty(k, np.float32)
    lib().orc_dequant(dtype, _ptr(row), k, _ptr(out))
    return out


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    w = np.ascontiguousarray(w, np.float32)
    y = np.empty_like(x)
    lib().orc_rms_norm(_ptr(x), _ptr(w), x.size, eps, _ptr(y))
    return y


def rope(v: np.ndarray, n_heads: int, pos: int, base: float, adjacent: bool) -> np.ndarray:
    v = np.array(v, dtype=np.float32, copy=True).reshape(-1)
    lib().orc_rope(_ptr(v), n_heads, v.size // n_heads, pos, base, int(adjacent))
    return v


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, t0: int, t1: int) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float32)
    K = np.ascontiguousarray(K, np.float32)
    V = np.ascontiguousarray(V, np.float32)
    o = np.empty(q.size, np.float32)
    lib().orc_attend(_ptr(q), _ptr(K), _ptr(V), q.size, t0, t1, _ptr(o))
    return o


ACT = {"silu": 0, "gelu": 1, "gelu_tanh": 2, "relu": 3}


def act(kind: str, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    y = np.empty_like(x)
    lib().orc_act(ACT[kind], _ptr(x), x.size, _ptr(y))
    return y


def matvec(dtype: int, W: np.ndarray, k: int, n: int, x: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W).view(np.uint8)
    x = np.ascontiguousarray(x, np.float32)
    y = np.empty(n, np.float32)
    lib().orc_matvec(dtype, _ptr(W), k, n, _ptr(x), _ptr(y))
    return y
