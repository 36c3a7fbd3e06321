"""decoder_token_step_gb300: the per-token forward of a GGUF decoder described by an .archdef text,
as a C-ABI CUDA library for GB300 (sm_103a) with a thin Python binding.

    from decoder_token_step_gb300 import build, syn
    build.build()                      # nvcc -> decoder_token_step_gb300/_build/libsyn.so
    m = syn.Model(syn.read_archdef("qwen3"), metadata, max_ctx=4096, arch="qwen3")
    m.load(name, dtype, ne, gguf_bytes) ...; m.finalize()
    logits, top = m.forward([token], pos)

Importing the package does not load the library; ``syn.lib()`` does, and raises if it is missing.
"""
from . import syn  # noqa: F401
