"""Python binding of libsyn (ctypes): argument marshalling only.

Every step of the forward runs in the CUDA library; this module converts Python / numpy / torch
arguments into the plain pointers and sizes of the C ABI (include/syn.h) and raises on error
statuses. There is no fallback: if the compiled library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Iterable, Optional, Tuple, Union

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsyn.so")

STATUS = {
    0: "SYN_OK", 1: "SYN_E_UNSUPPORTED_OP", 2: "SYN_E_SHAPE_MISMATCH", 3: "SYN_E_MISSING_TENSOR",
    4: "SYN_E_WEIGHT_FORMAT", 5: "SYN_E_OOM", 6: "SYN_E_BACKEND_INIT", 7: "SYN_E_INVALID_CONFIG",
    8: "SYN_E_ARCHDEF", 9: "SYN_E_CONTEXT_FULL", 10: "SYN_E_CUDA", 11: "SYN_E_STATE",
    12: "SYN_E_INVALID_ARG",
}
F32, F16, Q4_0, Q8_0 = 0, 1, 2, 8
TOKENS_ON_DEVICE, LOGITS_ON_DEVICE, ARGMAX_ON_DEVICE = 1, 2, 4


class SynError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.message = message


class Timings(ctypes.Structure):
    _fields_ = [("load_ms", ctypes.c_double), ("last_prefill_ms", ctypes.c_double),
                ("last_step_ms", ctypes.c_double), ("n_forward", ctypes.c_int64),
                ("n_launches", ctypes.c_int64), ("pool_bytes", ctypes.c_int64),
                ("kv_bytes", ctypes.c_int64), ("weight_bytes", ctypes.c_int64)]


_lib = None


def lib(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libsyn.so (built by ``decoder_token_step_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libsyn is not built ({p} missing): run decoder_token_step_gb300.build.build()")
    L = ctypes.CDLL(p)
    P, I, I64, S, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_char_p, ctypes.c_size_t
    sigs = {
        "syn_archdef_check": [S, S, SZ, P, P, SZ],
        "syn_create": [S, S, SZ, S, I, P, P],
        "syn_load_weights": [P, S, I, P, I, P, SZ],
        "syn_finalize": [P],
        "syn_reset_kv": [P],
        "syn_forward": [P, P, I, I, P, P, ctypes.c_uint],
        "syn_logits_device": [P, P, P],
        "syn_get_timings": [P, P],
        "syn_set_option": [P, S, I64],
        "syn_get_info": [P, S, P],
        "syn_debug_write_kv": [P, I, I, I, P, P],
        "syn_debug_read_kv": [P, I, I, I, P, P],
        "syn_debug_read_register": [P, S, P, I],
        "syn_debug_dequant": [P, S, I, I, P],
        "syn_get_profile": [P, P, SZ, I],
        "syn_archdef_sha256": [S, SZ, P],
        "syn_describe": [P, P, SZ],
        "syn_kv_create": [P, P],
        "syn_kv_select": [P, P],
        "syn_attention_static": [P, P, P, I, I, I, I, I, I, I, P, P],
        "syn_attention_static_status": [P],
    }
    for name, args in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.syn_last_error.argtypes = [P]
    L.syn_last_error.restype = S
    L.syn_destroy.argtypes = [P]
    L.syn_destroy.restype = None
    L.syn_kv_destroy.argtypes = [P]
    L.syn_kv_destroy.restype = None
    L.syn_debug_set_spin_limit.argtypes = [I]
    L.syn_debug_set_spin_limit.restype = None
    _lib = L
    return L


def archdef_check(text: str, arch: Optional[str] = None) -> int:
    """Validate an archdef text; returns its steps per layer or raises SynError."""
    err = ctypes.create_string_buffer(1024)
    steps = ctypes.c_int(0)
    b = text.encode()
    rc = lib().syn_archdef_check(arch.encode() if arch else None, b, len(b), ctypes.byref(steps), err, 1024)
    if rc:
        raise SynError(rc, err.value.decode())
    return steps.value


def archdef_sha256(text: str) -> str:
    """sha256 (hex) of a definition text, as the library identifies it."""
    b = text.encode()
    out = ctypes.create_string_buffer(65)
    rc = lib().syn_archdef_sha256(b, len(b), out)
    if rc:
        raise SynError(rc, "syn_archdef_sha256 failed")
    return out.value.decode()


def _ptr(x) -> int:
    """Data pointer of a numpy array or torch tensor (or an int address)."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"], "array must be contiguous"
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        assert x.is_contiguous(), "tensor must be contiguous"
        return x.data_ptr()
    raise TypeError(type(x))


def _on_device(x) -> bool:
    return hasattr(x, "is_cuda") and bool(x.is_cuda)


class Model:
    """One decoder: archdef text + GGUF metadata + weights + its KV cache."""

    def __init__(self, archdef_text: str, metadata: Union[Dict[str, str], str], max_ctx: int,
                 arch: Optional[str] = None, stream: Optional[int] = None):
        L = lib()
        md = metadata if isinstance(metadata, str) else "".join(f"{k}={v}\n" for k, v in metadata.items())
        h = ctypes.c_void_p()
        t = archdef_text.encode()
        rc = L.syn_create(arch.encode() if arch else None, t, len(t), md.encode(), int(max_ctx),
                          ctypes.c_void_p(stream or 0), ctypes.byref(h))
        self._h = h
        if rc:
            msg = L.syn_last_error(h).decode() if h.value else "allocation failed"
            self.close()
            raise SynError(rc, msg)
        self.max_ctx = int(max_ctx)

    # -------------------------------------------------------------- plumbing
    def _check(self, rc: int) -> None:
        if rc:
            raise SynError(rc, lib().syn_last_error(self._h).decode())

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().syn_destroy(self._h)
        self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -------------------------------------------------------------- load
    def load(self, name: str, dtype: int, ne: Iterable[int], data: np.ndarray) -> None:
        ne_a = (ctypes.c_int64 * len(tuple(ne)))(*ne)
        buf = np.ascontiguousarray(data).view(np.uint8).reshape(-1)
        self._check(lib().syn_load_weights(self._h, name.encode(), int(dtype), ne_a, len(ne_a),
                                           _ptr(buf), buf.nbytes))

    def load_tensors(self, tensors) -> None:
        for t in tensors.values() if isinstance(tensors, dict) else tensors:
            self.load(t.name, t.dtype, t.ne, t.data)

    def finalize(self) -> None:
        self._check(lib().syn_finalize(self._h))
        self.n_vocab = self.info("n_vocab")
        self.n_embd = self.info("n_embd")

    # -------------------------------------------------------------- run
    def reset_kv(self) -> None:
        self._check(lib().syn_reset_kv(self._h))

    def forward(self, tokens, pos: int, logits=None, argmax=None, want_logits: bool = True):
        """One forward over len(tokens) positions starting at `pos`.

        tokens: sequence / numpy int32 / torch int32 (host or cuda). logits / argmax: optional
        caller buffers (numpy or torch, host or cuda). With no buffers, returns host logits (and
        the greedy argmax) as numpy.
        """
        flags = 0
        if _on_device(tokens):
            flags |= TOKENS_ON_DEVICE
            tok = tokens
            n = tokens.numel()
        else:
            tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32).reshape(-1))
            n = tok.size
        ret_logits = None
        if logits is None and want_logits:
            logits = ret_logits = np.empty(self.n_vocab, np.float32)
        if logits is not None and _on_device(logits):
            flags |= LOGITS_ON_DEVICE
        ret_arg = None
        if argmax is None and ret_logits is not None:
            argmax = ret_arg = np.zeros(1, np.int32)
        if argmax is not None and _on_device(argmax):
            flags |= ARGMAX_ON_DEVICE
        self._check(lib().syn_forward(self._h, _ptr(tok), int(n), int(pos), _ptr(logits), _ptr(argmax), flags))
        if ret_logits is not None:
            return ret_logits, int(ret_arg[0]) if ret_arg is not None else None
        return None

    def forward_raw(self, tokens_ptr: int, n: int, pos: int, logits_ptr: int, argmax_ptr: int, flags: int) -> None:
        """Direct C-ABI call with raw pointers (device-resident loops)."""
        self._check(lib().syn_forward(self._h, tokens_ptr, n, pos, logits_ptr, argmax_ptr, flags))

    def logits_device(self) -> Tuple[int, int]:
        p = ctypes.c_void_p()
        n = ctypes.c_int()
        self._check(lib().syn_logits_device(self._h, ctypes.byref(p), ctypes.byref(n)))
        return p.value, n.value

    # -------------------------------------------------------------- options / info
    def set_option(self, key: str, value: int) -> None:
        self._check(lib().syn_set_option(self._h, key.encode(), int(value)))

    def describe(self) -> Dict[str, str]:
        """The model's status line as a dict (architecture, steps, definition sha256, shapes...)."""
        buf = ctypes.create_string_buffer(4096)
        self._check(lib().syn_describe(self._h, buf, len(buf)))
        return dict(kv.split("=", 1) for kv in buf.value.decode().split())

    def new_kv(self) -> "KvCache":
        """A second conversation on this model: its own KV cache (select it with select_kv)."""
        return KvCache(self)

    def select_kv(self, kv: Optional["KvCache"]) -> None:
        """Make kv (or, with None, the model's own cache) the conversation that forwards,
        resets and KV reads/writes act on."""
        self._check(lib().syn_kv_select(self._h, kv._h if kv is not None else None))

    def info(self, key: str) -> int:
        v = ctypes.c_int64()
        self._check(lib().syn_get_info(self._h, key.encode(), ctypes.byref(v)))
        return v.value

    def timings(self) -> Dict[str, float]:
        t = Timings()
        self._check(lib().syn_get_timings(self._h, ctypes.byref(t)))
        return {f: getattr(t, f) for f, _ in Timings._fields_}

    def profile(self, reset: bool = True) -> Dict[str, Dict[str, float]]:
        """Per-kind device time of the forwards run with option "profile" = 1."""
        buf = ctypes.create_string_buffer(1 << 16)
        self._check(lib().syn_get_profile(self._h, buf, len(buf), int(reset)))
        out = {}
        for line in buf.value.decode().splitlines():
            kind, launches, ms, nbytes, flops = line.split()
            out[kind] = {"launches": int(launches), "ms": float(ms), "bytes": float(nbytes), "flops": float(flops)}
        return out

    # -------------------------------------------------------------- test support
    def write_kv(self, layer: int, pos0: int, k: np.ndarray, v: np.ndarray) -> None:
        k = np.ascontiguousarray(k, np.float32)
        v = np.ascontiguousarray(v, np.float32)
        self._check(lib().syn_debug_write_kv(self._h, layer, pos0, k.shape[1], _ptr(k), _ptr(v)))

    def read_kv(self, layer: int, pos0: int, n: int, n_head_kv: int, head_dim: int):
        k = np.empty((n_head_kv, n, head_dim), np.float32)
        v = np.empty_like(k)
        self._check(lib().syn_debug_read_kv(self._h, layer, pos0, n, _ptr(k), _ptr(v)))
        return k, v

    def read_register(self, name: str, count: int) -> np.ndarray:
        out = np.empty(count, np.float32)
        self._check(lib().syn_debug_read_register(self._h, name.encode(), _ptr(out), count))
        return out

    def dequant(self, name: str, row0: int, nrows: int, k: int) -> np.ndarray:
        out = np.empty((nrows, k), np.float32)
        self._check(lib().syn_debug_dequant(self._h, name.encode(), row0, nrows, _ptr(out)))
        return out


def archdef_path(arch: str) -> str:
    return os.path.join(_HERE, "archdefs", arch + ".archdef")


def read_archdef(arch: str) -> str:
    with open(archdef_path(arch)) as f:
        return f.read()


class KvCache:
    """One conversation's KV cache on a loaded model (syn_kv_create / syn_kv_destroy)."""

    def __init__(self, model: Model):
        h = ctypes.c_void_p()
        model._check(lib().syn_kv_create(model._h, ctypes.byref(h)))
        self._h = h.value
        self._model = model

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().syn_kv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
