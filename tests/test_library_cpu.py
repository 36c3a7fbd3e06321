"""The C-ABI library on the CPU: it builds, loads, exports every symbol of include/syn.h, and its
archdef parser behaves as "Local inference and architectures" (synsema.dev) describes. No GPU."""
import ctypes
import json
import os
import re

import pytest

from decoder_token_step_gb300 import build as syn_build
from decoder_token_step_gb300 import syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden", "archdef_facts.json")


@pytest.fixture(scope="module", autouse=True)
def built():
    syn_build.build()


def facts():
    with open(GOLDEN) as f:
        return json.load(f)


def header_symbols():
    with open(os.path.join(ROOT, "include", "syn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(syn_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = header_symbols()
    assert len(names) >= 15
    L = ctypes.CDLL(syn.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_library_is_compiled_for_sm_103a_only():
    assert syn_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-lineinfo" in syn_build._flags()


@pytest.mark.parametrize("arch", ["gemma3", "llama", "qwen2", "qwen3"])
def test_shipped_definitions_have_the_published_step_counts(arch):
    assert syn.archdef_check(syn.read_archdef(arch), arch) == facts()["steps_per_layer"][arch]


def _statements(text, section):
    out, cur = [], None
    for raw in text.split("\n"):
        s = raw.split("#")[0].strip()
        if s in ("prologue", "block", "epilogue"):
            cur = s
            continue
        if not s or cur != section:
            continue
        m = re.match(r"^(?:(\w+)\s*=\s*)?(\w+)\((.*)\)$", s)
        dst, op, args = m.group(1), m.group(2), [a.strip() for a in m.group(3).split(",")]
        out.append([dst or args[0], op, args if dst else args])
    return out


def test_shipped_qwen3_matches_the_printed_definition():
    text = syn.read_archdef("qwen3")
    f = facts()["qwen3"]
    for sec in ("prologue", "block", "epilogue"):
        assert _statements(text, sec) == [[d, o, a] for d, o, a in f[sec]]


def test_qwen2_is_llama_plus_three_bias_lines():
    l2 = _statements(syn.read_archdef("qwen2"), "block")
    ll = _statements(syn.read_archdef("llama"), "block")
    assert [s for s in l2 if s[1] != "add_bias"] == ll
    assert [s[2][0] for s in l2 if s[1] == "add_bias"] == ["q", "k", "v"]


def test_typo_names_line_28_and_suggests_the_fix():
    f = facts()["typo"]
    text = syn.read_archdef("qwen3").replace("  silu(g)", "  siluu(g)")
    with pytest.raises(syn.SynError) as e:
        syn.archdef_check(text, "qwen3")
    assert e.value.status == 8
    assert e.value.message == (f"qwen3.archdef: line {f['line']}: unknown operation `{f['written']}`"
                               f" — did you mean `{f['suggested']}`?")


@pytest.mark.parametrize("case,edit,expected", [
    ("section", ("block\n", "blok\n"), "unknown section or operation `blok` — did you mean `block`?"),
    ("param", ("kind decoder", "kind decoder\nparam window_patern 6"),
     "unknown param `window_patern` (known: window_pattern, rope_pairs) — did you mean `window_pattern`?"),
    ("kind", ("kind decoder", "kind decodr"), "only `kind decoder` is supported — did you mean `decoder`?"),
    ("register", ("  add(x, d)", "  add(x, dd)"), "register `dd` is read before it is assigned — did you mean `d`?"),
    ("rope_pairs", ("param rope_pairs adjacent", "param rope_pairs adjacnt"),
     "rope_pairs must be `adjacent` or `half` — did you mean `adjacent`?"),
    ("far", ("  add(x, d)", "  add(x, zzzz)"), "register `zzzz` is read before it is assigned"),
])
def test_parse_errors_name_the_line_and_suggest_the_nearest_word(case, edit, expected):
    """Every parse error that a typo can cause names its line and, when a known word is within two
    edits, suggests it (and only then)."""
    base = syn.read_archdef("llama")
    assert edit[0] in base
    text = base.replace(edit[0], edit[1], 1)
    with pytest.raises(syn.SynError) as e:
        syn.archdef_check(text, "llama")
    assert e.value.status == 8
    assert re.match(r"^llama\.archdef: line \d+: ", e.value.message)
    assert e.value.message.split(": ", 2)[2] == expected, e.value.message


# The pages name nine of the twenty-one rejected words; the other twelve are the parser's reading
# (control flow and I/O words of common languages).
EXTRA_WORDS = ["else", "return", "def", "fn", "let", "call", "include", "exit", "system", "socket",
               "file", "load"]


def test_twenty_one_control_flow_and_io_words_are_unknown_ops():
    f = facts()
    words = f["rejected_words_named"] + EXTRA_WORDS
    assert len(set(words)) == f["rejected_word_count"] == 21
    base = syn.read_archdef("llama")
    for w in words:
        for line in (f"  {w}(x)", f"  x = {w}(x)"):
            text = base.replace("  add(x, d)", line + "\n  add(x, d)")
            with pytest.raises(syn.SynError) as e:
                syn.archdef_check(text, "llama")
            assert f"unknown operation `{w}`" in e.value.message, (w, e.value.message)


def test_sixteen_ops_are_the_vocabulary():
    ops = facts()["operations"]
    assert len(ops) == 16
    base = syn.read_archdef("llama")
    # every op name is accepted as an op (arity errors are fine, "unknown operation" is not)
    for op in ops:
        text = base.replace("  add(x, d)", f"  {op}(x)\n  add(x, d)")
        try:
            syn.archdef_check(text, "llama")
        except syn.SynError as e:
            assert "unknown operation" not in e.message


def test_file_name_must_match_arch_line():
    with pytest.raises(syn.SynError, match="declares `arch qwen3`; the file name says `llama`"):
        syn.archdef_check(syn.read_archdef("qwen3"), "llama")


@pytest.mark.parametrize("mutation, fragment", [
    (lambda t: t.replace("\nblock\n", "\nepilogue\n  x = last(x)\nblock\n", 1), "out of order"),
    (lambda t: t.replace("a = attention(q, k, v)", "a = attention(q, k)"), "takes 3 argument"),
    (lambda t: t.replace("o = matmul(a, blk", "o = matmul(zz, blk"), "read before it is assigned"),
    (lambda t: t.replace("kind decoder", "kind encoder"), "kind decoder"),
    (lambda t: t.replace("arch qwen3\n", ""), "missing `arch"),
    (lambda t: t + "\nparam colour blue\n", "param"),
    (lambda t: t.replace("  x = embed(token_embd.weight)", "  embed(x)"), "needs a destination"),
])
def test_malformed_definitions_fail_early_with_the_line(mutation, fragment):
    with pytest.raises(syn.SynError) as e:
        syn.archdef_check(mutation(syn.read_archdef("qwen3")), "qwen3")
    assert fragment in e.value.message
    assert e.value.message.startswith("qwen3.archdef: line ")


def test_comments_and_blank_lines_are_free():
    text = syn.read_archdef("llama")
    noisy = "\n\n# a comment\n".join(text.split("\n"))
    assert syn.archdef_check(noisy, "llama") == 16


def test_create_without_a_gpu_reports_backend_init():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import synth
    cfg = synth.CONFIGS["tiny"]
    with pytest.raises(syn.SynError) as e:
        syn.Model(syn.read_archdef("qwen3"), synth.metadata(cfg), 64, arch="qwen3")
    assert e.value.status == 6


def test_create_rejects_a_broken_definition_before_touching_the_device():
    import synth
    text = syn.read_archdef("qwen3").replace("  silu(g)", "  siluu(g)")
    with pytest.raises(syn.SynError) as e:
        syn.Model(text, synth.metadata(synth.CONFIGS["tiny"]), 64, arch="qwen3")
    assert e.value.status == 8 and "line 28" in e.value.message


@pytest.mark.parametrize("key,value,fragment", [
    ("qwen3.block_count", "", "not a 32-bit integer"),
    ("qwen3.block_count", "4294967298", "not a 32-bit integer"),        # would wrap to 2 as an int
    ("qwen3.block_count", "2x", "not a 32-bit integer"),
    ("qwen3.block_count", "0", "must be positive"),
    ("qwen3.attention.head_count_kv", "3", "multiple of head_count_kv"),
    ("qwen3.attention.layer_norm_rms_epsilon", "nan", "not a finite number"),
    ("qwen3.attention.layer_norm_rms_epsilon", "", "not a finite number"),
    ("qwen3.attention.layer_norm_rms_epsilon", "-1e-6", "must be >= 0"),
    ("qwen3.rope.freq_base", "inf", "not a finite number"),
    ("qwen3.rope.freq_base", "0", "freq_base > 0"),
    ("qwen3.attention.sliding_window", "-5", "sliding_window >= 0"),
])
def test_create_refuses_bad_metadata_before_touching_the_device(key, value, fragment):
    """GGUF metadata is checked when the model is created: an empty, non-numeric, out-of-range or
    non-finite value, or an impossible head layout, is SYN_E_INVALID_CONFIG naming the key, never a
    silently truncated or NaN setting."""
    import synth
    md = synth.metadata(synth.CONFIGS["tiny"])
    assert key in md or key.endswith("sliding_window")
    md[key] = value
    with pytest.raises(syn.SynError) as e:
        syn.Model(syn.read_archdef("qwen3"), md, 64, arch="qwen3")
    assert e.value.status == 7 and fragment in e.value.message, e.value.message


@pytest.mark.parametrize("factor,accepted", [("2.5", True), ("embedding_length", True), ("head_count", True),
                                             ("embeding_length", False), ("nan", False), ("2.5x", False)])
def test_scale_factor_is_a_number_or_a_metadata_key(factor, accepted):
    """`scale(x, c)`: c is a float literal or the name of a GGUF metadata key (read under the
    architecture's prefix); a misspelt key or a non-finite value is refused at creation with its
    line, never read as 0."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import synth
    text = syn.read_archdef("qwen3").replace("  x = embed(token_embd.weight)\n",
                                             f"  x = embed(token_embd.weight)\n  scale(x, {factor})\n", 1)
    assert f"scale(x, {factor})" in text
    with pytest.raises(syn.SynError) as e:
        syn.Model(text, synth.metadata(synth.CONFIGS["tiny"]), 64, arch="qwen3")
    if accepted:
        assert e.value.status == 6                                  # got as far as the device check
    else:
        assert e.value.status == 8 and "line 11" in e.value.message and factor in e.value.message


def test_create_refuses_unsupported_head_layouts():
    import synth
    for over, fragment in (({"qwen3.attention.key_length": "96"}, "head_dim 96"),
                           ({"qwen3.attention.head_count": "36", "qwen3.attention.head_count_kv": "4"},
                            "too many query heads")):
        md = synth.metadata(synth.CONFIGS["tiny"])
        md.update(over)
        with pytest.raises(syn.SynError) as e:
            syn.Model(syn.read_archdef("qwen3"), md, 64, arch="qwen3")
        assert e.value.status == 1 and fragment in e.value.message, e.value.message


# ------------------------------------------------------------------------------ definition identity

def test_archdef_sha256_matches_the_standard_vectors_and_hashlib():
    """The library's SHA-256 (written from FIPS 180-4) against the standard's short-message vectors
    and Python's hashlib, including lengths around the one- and two-block padding boundaries."""
    import hashlib
    assert syn.archdef_sha256("") == "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855"
    assert syn.archdef_sha256("abc") == "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"
    assert syn.archdef_sha256("abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq") == \
        "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1"
    for n in (55, 56, 57, 63, 64, 65, 119, 120, 1000):
        t = "".join(chr(97 + (i * 7) % 26) for i in range(n))
        assert syn.archdef_sha256(t) == hashlib.sha256(t.encode()).hexdigest(), n
    for arch in ("qwen3", "llama", "qwen2", "gemma3"):
        text = syn.read_archdef(arch)
        assert syn.archdef_sha256(text) == hashlib.sha256(text.encode()).hexdigest()


def _header_params():
    """name -> list of parameter declarations, from the C prototypes in include/syn.h."""
    with open(os.path.join(ROOT, "include", "syn.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(syn_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = [p.strip() for p in m.group(2).split(",") if p.strip()]
        out[m.group(1)] = [] if params == ["void"] else params
    return out


def _ctype_for(decl):
    """The ctypes type a parameter declaration needs in the binding."""
    if "*" in decl:
        return (ctypes.c_void_p, ctypes.c_char_p)
    base = decl.rsplit(" ", 1)[0].replace("const ", "").strip()
    return {"int": (ctypes.c_int,), "int64_t": (ctypes.c_int64,), "size_t": (ctypes.c_size_t,),
            "unsigned": (ctypes.c_uint,), "syn_dtype": (ctypes.c_int,)}[base]


def test_binding_marshals_every_call_as_the_header_declares():
    """Every function the Python binding types has the header's parameter count, and each argument
    goes across as a pointer where the header has one and as an integer of the declared width
    elsewhere."""
    params = _header_params()
    L = syn.lib()
    typed = 0
    for name, decls in params.items():
        f = getattr(L, name)
        if f.argtypes is None:
            continue   # not used from Python (the tests that call it set its types themselves)
        typed += 1
        assert len(f.argtypes) == len(decls), (name, decls)
        for t, d in zip(f.argtypes, decls):
            assert t in _ctype_for(d), (name, d, t)
    assert typed >= 20


def test_timings_struct_matches_the_header_field_by_field():
    """syn_timings crosses the ABI by value: the binding's ctypes structure has the header's fields,
    in order, with the same types (so the same offsets)."""
    with open(os.path.join(ROOT, "include", "syn.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    body = re.search(r"typedef struct\s*\{([^}]*)\}\s*syn_timings\s*;", text).group(1)
    fields = [tuple(d.split()) for d in (x.strip() for x in body.split(";")) if d]
    ctype = {"double": ctypes.c_double, "int64_t": ctypes.c_int64}
    assert [(n, ctype[t]) for t, n in fields] == list(syn.Timings._fields_)


_FUZZ = r'''
import random, sys
sys.path.insert(0, sys.argv[1])
from decoder_token_step_gb300 import syn
base = syn.read_archdef("qwen3")
rng = random.Random(7)
alphabet = list("abcdefghijklmnopqrstuvwxyz_.0123456789(){}|=,#\t \n") + ["é", "\x00", "\x7f", "\r"]
words = ["embed", "rms_norm", "matmul", "attention", "block", "epilogue", "prologue", "param", "arch", "kind",
         "x", "q", "{i}", "blk.{i}.attn_q.weight", "|", "last", "silu", "mul", "if", "while", "rope"]
ok = bad = 0
for it in range(3000):
    t = base
    for _ in range(rng.randint(1, 4)):
        op, lines = rng.randrange(7), t.split("\n")
        if op == 0 and t:
            i = rng.randrange(len(t)); t = t[:i] + t[i + 1:]
        elif op == 1:
            i = rng.randrange(len(t) + 1); t = t[:i] + rng.choice(alphabet) + t[i:]
        elif op == 2:
            i = rng.randrange(len(lines)); lines.insert(i, lines[i]); t = "\n".join(lines)
        elif op == 3:
            del lines[rng.randrange(len(lines))]; t = "\n".join(lines)
        elif op == 4:
            i, j = rng.randrange(len(lines)), rng.randrange(len(lines)); lines[i], lines[j] = lines[j], lines[i]
            t = "\n".join(lines)
        elif op == 5:
            t = t[:rng.randrange(len(t) + 1)]
        else:
            toks = t.split(" "); toks[rng.randrange(len(toks))] = rng.choice(words); t = " ".join(toks)
    try:
        syn.archdef_check(t, "qwen3"); ok += 1
    except syn.SynError as e:
        assert e.status == 8 and e.message.startswith("qwen3.archdef: line "), (repr(t), e.status, e.message)
        bad += 1
print(ok, bad)
'''


def test_randomly_mutated_definitions_are_accepted_or_refused_with_a_line_never_crash():
    """3000 seeded random edits of the qwen3 text (characters deleted or inserted, NUL and non-ASCII
    included; lines duplicated, deleted or swapped; truncation; words replaced by op, section and
    register names): the parser returns SYN_OK or SYN_E_ARCHDEF with a line number, and the process
    survives (it runs in a child process, so a crash fails the test instead of ending the run)."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", _FUZZ, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    ok, bad = map(int, r.stdout.split())
    assert ok + bad == 3000 and bad > 2000


def test_every_call_refuses_null_arguments_without_touching_anything():
    """Every status-returning entry point of the binding, called with NULL pointers and zero sizes,
    returns SYN_E_INVALID_ARG ("Execution contract", section "Error semantics": errors are values,
    the process never aborts); syn_destroy and syn_kv_destroy accept NULL; syn_last_error(NULL)
    still returns a message. syn_attention_static_status takes only a stream, for which NULL is the
    legacy default stream (a valid argument), so it is not among them."""
    L = syn.lib()
    called = 0
    for name, decls in _header_params().items():
        f = getattr(L, name)
        if f.argtypes is None or f.restype is not ctypes.c_int or name == "syn_attention_static_status":
            continue
        args = [None if t in (ctypes.c_void_p, ctypes.c_char_p) else 0 for t in f.argtypes]
        assert f(*args) == 12, name
        called += 1
    assert called >= 19
    L.syn_destroy(None)
    L.syn_kv_destroy(None)
    assert L.syn_last_error(None)


def test_the_binding_fails_loudly_when_the_library_is_missing(monkeypatch, tmp_path):
    """No fallback: without libsyn.so the binding raises at the first call instead of computing
    anything some other way."""
    import synth
    monkeypatch.setattr(syn, "_lib", None)
    monkeypatch.setattr(syn, "LIB_PATH", str(tmp_path / "libsyn.so"))
    with pytest.raises(ImportError, match="not built"):
        syn.Model(syn.read_archdef("qwen3"), synth.metadata(synth.CONFIGS["tiny"]), 64, arch="qwen3")
    with pytest.raises(ImportError):
        syn.archdef_check(syn.read_archdef("qwen3"), "qwen3")


def test_the_metadata_of_every_workload_passes_validation():
    """The checks on GGUF metadata refuse no real configuration: each workload's metadata (and a
    windowed variant) gets past them to the device check (SYN_E_BACKEND_INIT on a machine without a
    GPU)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import synth
    for name, cfg in synth.CONFIGS.items():
        for c in (cfg, synth.scaled(cfg, sliding_window=37)):
            with pytest.raises(syn.SynError) as e:
                syn.Model(syn.read_archdef(c.arch), synth.metadata(c, 128), 128, arch=c.arch)
            assert e.value.status == 6, (name, e.value.message)
