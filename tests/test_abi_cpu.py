"""The C-ABI library builds, loads and exports every symbol include/pkv.h
declares; host-side sizing and validation behave as documented (CPU only: no
kernel is launched)."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_attention_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def _declared_symbols():
    names = []
    for h in HEADERS:
        src = open(h).read()
        names += re.findall(r"PKV_API\s+[\w\s\*]*?\b(pkv_\w+)\s*\(", src)
    return names


def test_header_declares_the_three_operations():
    names = _declared_symbols()
    for op in ("pkv_reshape_and_cache", "pkv_paged_decode", "pkv_varlen_prefill"):
        assert op in names


def test_library_exports_every_declared_symbol():
    lib = pkv.load_library()
    declared = _declared_symbols()
    assert declared, "no PKV_API declarations found"
    for name in declared:
        assert hasattr(lib, name), f"libpkv.so does not export {name}"
    assert set(pkv.EXPORTED_SYMBOLS) <= set(declared)


def test_status_strings_and_version():
    lib = pkv.load_library()
    assert lib.pkv_version() >= 100
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(3) == b"PKV_ERR_WORKSPACE"
    assert lib.pkv_status_string(5) == b"PKV_ERR_OUT_OF_RANGE"
    assert lib.pkv_status_string(6) == b"PKV_ERR_TIMEOUT"
    assert lib.pkv_status_string(99) == b"PKV_ERR_UNKNOWN"


def test_decode_workspace_size_grows_with_partitions():
    a = pkv.paged_decode_workspace_size(64, 32, 128, 4096, 512)
    b = pkv.paged_decode_workspace_size(64, 32, 128, 8192, 512)
    assert b > a
    # split-KV partials: B * Hq * P * (D + 1) floats, 256-byte rounded
    assert a >= 64 * 32 * 8 * 129 * 4
    # a window bounds the partitions a sequence can touch
    w = pkv.paged_decode_workspace_size(8, 64, 64, 131072, 512, 127)
    assert w <= 8 * 64 * 2 * 65 * 4 + 1024


# ---------------------------------------------------------------------------
# host validation: every case below is rejected before any CUDA call.  The
# pointers are fake, so these run only where no GPU is present.
# ---------------------------------------------------------------------------
nogpu = pytest.mark.skipif(torch.cuda.is_available(),
                           reason="fake-pointer validation tests run without a GPU only")
FAKE = 0x10000  # 256-byte aligned, never dereferenced


def _desc(nb=64, bs=16, hkv=8, d=128, dtype=1):
    return pkv.CacheDesc(nb, bs, hkv, d, dtype)


def _decode(lib, desc=None, batch=4, hq=32, window=-1, part=512, ws_bytes=1 << 30,
            ws=FAKE, q=FAKE, max_blocks=8, max_seqlen=128, scale=0.1):
    return lib.pkv_paged_decode(FAKE, q, FAKE, FAKE, desc or _desc(), FAKE, max_blocks, FAKE,
                                max_seqlen, None, None, batch, hq, window, scale, part, None, ws,
                                ws_bytes, None, None)


@nogpu
@pytest.mark.parametrize("kw,expected", [
    (dict(desc=_desc(d=72)), 2),                 # head_dim without a kernel
    (dict(desc=_desc(d=512)), 2),
    (dict(desc=_desc(d=256, dtype=0)), 2),       # fp32 decode stops at 128
    (dict(desc=_desc(bs=8)), 2),                 # block size without a kernel
    (dict(desc=_desc(dtype=7)), 2),              # unknown dtype
    (dict(desc=_desc(nb=0)), 1),                 # empty pool
    (dict(desc=_desc(nb=1 << 28)), 2),           # pool rows beyond int32
    (dict(hq=30), 1),                            # Hq % Hkv != 0
    (dict(hq=8 * 17), 2),                        # group of 17
    (dict(part=500), 1),                         # partition not a multiple of the page
    (dict(part=32768), 1),                       # partition above the maximum
    (dict(window=-2), 1),                        # bad window
    (dict(batch=-1), 1),
    (dict(max_blocks=0), 1),
    (dict(scale=float("nan")), 1),
    (dict(ws=None), 3),                          # no workspace
    (dict(ws=FAKE + 16), 3),                     # misaligned workspace
    (dict(ws_bytes=1000), 3),                    # too small
    (dict(q=FAKE + 2), 1),                       # misaligned q
    (dict(batch=0), 0),                          # nothing to do
])
def test_decode_validation(kw, expected):
    assert _decode(pkv.load_library(), **kw) == expected


@nogpu
def test_reshape_and_cache_validation():
    lib = pkv.load_library()
    f = lib.pkv_reshape_and_cache
    bad_layout = _desc()
    bad_layout.layout = 2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, bad_layout, None, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 0, _desc(), None, None) == 0
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, _desc(), None, None) == 1
    assert f(None, FAKE, FAKE, FAKE, FAKE, 3, _desc(), None, None) == 1
    assert f(FAKE + 4, FAKE, FAKE, FAKE, FAKE, 3, _desc(), None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, _desc(dtype=3), None, None) == 2
    # fp32 rows of 3 heads x 4 dims = 48 bytes are fine; bf16 rows of 3 x 2 = 12 bytes are not
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, _desc(hkv=3, d=2, dtype=1), None, None) == 2


@nogpu
@pytest.mark.parametrize("change,expected", [
    (dict(window=-2), 1),
    (dict(d=512), 2),               # no prefill kernel for head_dim 512
    (dict(d=72), 2),
    (dict(dtype=0), 2),             # fp32 prefill not in this version
    (dict(hq=24), 2),               # group of 3 (not a power of two)
    (dict(total_q=0), 0),
    (dict(ws_bytes=16), 3),
    (dict(max_ctas=-1), 1),         # a negative CTA cap
])
def test_prefill_validation(change, expected):
    lib = pkv.load_library()
    a = dict(causal=1, dtype=1, hq=32, total_q=100, ws_bytes=1 << 30, window=-1, d=128,
             max_ctas=0)
    a.update(change)
    st = lib.pkv_varlen_prefill(FAKE, FAKE, FAKE, FAKE, _desc(dtype=a["dtype"], d=a["d"]), FAKE,
                                8, FAKE,
                                FAKE, 64, 128, a["total_q"], None, None, 2, a["hq"], a["causal"],
                                a["window"], 0.1, None, FAKE, a["ws_bytes"], a["max_ctas"], None,
                                None)
    assert st == expected


@nogpu
@pytest.mark.parametrize("change,expected", [
    (dict(total_k=-1), 1),
    (dict(hkv=0), 1),
    (dict(dtype=3), 2),
    (dict(dtype=0), 2),             # fp32 prefill not in this version
    (dict(d=72), 2),                # not a multiple of 16
    (dict(d=512), 2),               # no kernel for head_dim 512
    (dict(hq=24), 2),               # group of 3 (not a power of two)
    (dict(hq=12), 1),               # not a multiple of num_kv_heads
    (dict(k=None), 1),              # keys missing although total_k > 0
    (dict(k=FAKE + 8), 1),          # not 16-byte aligned
    (dict(total_q=0), 0),
    (dict(ws_bytes=16), 3),
])
def test_prefill_contiguous_validation(change, expected):
    lib = pkv.load_library()
    a = dict(total_k=500, hkv=8, d=128, dtype=1, hq=32, total_q=100, ws_bytes=1 << 30, k=FAKE)
    a.update(change)
    st = lib.pkv_varlen_prefill_contiguous(
        FAKE, FAKE, a["k"], FAKE, a["total_k"], a["hkv"], a["d"], a["dtype"], FAKE, FAKE, 64,
        128, a["total_q"], None, None, 2, a["hq"], 1, -1, 0.1, None, FAKE, a["ws_bytes"], None,
        None)
    assert st == expected


def test_binding_rejects_cpu_tensors():
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.paged_decode(q, kc, kc, torch.zeros(2, 1, dtype=torch.int32),
                         torch.zeros(2, dtype=torch.int32), max_seqlen=16)


@nogpu
@pytest.mark.parametrize("change,expected", [
    (dict(num_tokens=0), 0),
    (dict(num_tokens=-1), 1),
    (dict(rd=0), 1),
    (dict(rd=130), 1),              # longer than head_dim
    (dict(rd=7), 1),                # odd
    (dict(rd=24), 2),               # bf16 needs a multiple of 16
    (dict(max_pos=0), 1),
    (dict(query=None), 1),          # query missing with num_qo_heads > 0
    (dict(query=None, hq=0), 4),    # valid; no device to launch on here
    (dict(table=FAKE + 8), 1),      # not 16-byte aligned
    (dict(dtype=3), 2),
])
def test_rope_reshape_and_cache_validation(change, expected):
    lib = pkv.load_library()
    a = dict(num_tokens=10, rd=64, max_pos=4096, query=FAKE, hq=32, table=FAKE, dtype=1)
    a.update(change)
    st = lib.pkv_rope_reshape_and_cache(a["query"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                        a["num_tokens"], a["hq"], _desc(dtype=a["dtype"]),
                                        a["table"], a["max_pos"], a["rd"], 1, None, None)
    if expected == 4:
        assert st != 0 and st not in (1, 2, 3)
    else:
        assert st == expected


@nogpu
def test_rope_table_validation():
    f = pkv.load_library().pkv_rope_cos_sin_table
    assert f(FAKE, 0, 64, 10000.0, 1.0, 1.0, None) == 0       # nothing to fill
    assert f(FAKE, 10, 63, 10000.0, 1.0, 1.0, None) == 1      # odd rotary_dim
    assert f(FAKE, 10, 64, -1.0, 1.0, 1.0, None) == 1         # base must be positive
    assert f(FAKE, 10, 64, 10000.0, 0.0, 1.0, None) == 1      # scale must be positive
    assert f(FAKE, 10, 64, 10000.0, 1.0, 0.0, None) == 1      # ntk_alpha must be positive
    assert f(FAKE, 10, 2, 10000.0, 1.0, 2.0, None) == 1       # NTK needs rotary_dim > 2
    assert f(FAKE, 0, 2, 10000.0, 1.0, 1.0, None) == 0        # rotary_dim 2 without NTK
    assert f(None, 10, 64, 10000.0, 1.0, 1.0, None) == 1


@nogpu
def test_get_device_error_validation():
    assert pkv.load_library().pkv_get_device_error(None, None, 0, None) == 1
    # the bounded-wait self-test needs an error word to report into
    assert pkv.load_library().pkv_selftest_bounded_wait(None, None) == 1


# ---------------------------------------------------------------------------
# the binding against the header: ctypes passes arguments by the declared
# types, so a declaration that drifts from include/pkv.h would pass wrong
# values without any error
# ---------------------------------------------------------------------------
def _strip_c_comments(src):
    return re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", src, flags=re.S))


def _prototypes():
    """(name, return type, [parameter types]) of every PKV_API function."""
    out = []
    for h in HEADERS:
        src = _strip_c_comments(open(h).read())
        for ret, name, params in re.findall(
                r"PKV_API\s+([\w\s\*]*?)\s*\b(pkv_\w+)\s*\(([^)]*)\)\s*;", src):
            ps = [" ".join(p.split()) for p in params.split(",")]
            if ps == ["void"]:
                ps = []
            out.append((name, " ".join(ret.split()), ps))
    return out


_C_TYPES = {"int": ctypes.c_int, "int32_t": ctypes.c_int32, "pkv_status": ctypes.c_int,
            "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t, "float": ctypes.c_float,
            "double": ctypes.c_double, "pkv_cache_desc": pkv.CacheDesc}


def _ctype(decl, is_return=False):
    """The ctypes type a C declaration (type, optionally followed by a name) maps to."""
    if "*" in decl:
        if is_return and decl.replace(" ", "") == "constchar*":
            return ctypes.c_char_p
        return ctypes.c_void_p
    words = [w for w in decl.split() if w != "const"]
    base = words[0] if is_return else " ".join(words[:-1])
    return _C_TYPES[base]


def test_binding_declares_every_function_as_the_header_does():
    lib = pkv.load_library()
    protos = _prototypes()
    assert {n for n, _, _ in protos} == set(_declared_symbols())
    for name, ret, params in protos:
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes in the binding"
        want = [_ctype(p) for p in params]
        assert list(fn.argtypes) == want, f"{name}: argtypes differ from the header"
        assert fn.restype is _ctype(ret, is_return=True), f"{name}: restype differs"


def test_cache_desc_matches_the_header_struct():
    src = _strip_c_comments(open(os.path.join(ROOT, "include", "pkv.h")).read())
    body = re.search(r"typedef struct pkv_cache_desc\s*\{(.*?)\}\s*pkv_cache_desc;", src,
                     re.S).group(1)
    fields = [f.split() for f in body.split(";") if f.strip()]
    assert [(n, _C_TYPES[t]) for t, n in fields] == list(pkv.CacheDesc._fields_)


def test_python_sources_define_every_name_they_read():
    """A static check over the package, the bench, the entry points, the
    oracle's loader and the tests: every global name a function reads is
    defined in its module or is a builtin."""
    import builtins
    import glob
    import symtable
    files = (glob.glob(os.path.join(ROOT, "paged_kv_cache_attention_gb300", "*.py")) +
             glob.glob(os.path.join(ROOT, "tests", "*.py")) +
             [os.path.join(ROOT, f) for f in ("bench.py", "__graft_entry__.py",
                                              os.path.join("oracle", "__init__.py"))])
    missing = []
    for path in files:
        top = symtable.symtable(open(path).read(), path, "exec")
        known = set(top.get_identifiers()) | set(dir(builtins))

        def walk(t):
            for s in t.get_symbols():
                if s.is_global() and not s.is_declared_global() and s.get_name() not in known:
                    missing.append(f"{os.path.relpath(path, ROOT)}: {t.get_name()} reads "
                                   f"{s.get_name()}")
            for c in t.get_children():
                walk(c)
        walk(top)
    assert not missing, "\n".join(missing)


@nogpu
def test_noalloc_rejects_problems_beyond_the_scratch_before_any_cuda_call():
    lib = pkv.load_library()
    huge = 1 << 20  # 2048 partitions of 512 for 4 x 32 heads: more than the 32 MiB scratch
    assert pkv.paged_decode_workspace_size(4, 32, 128, huge, 512, -1) > (32 << 20)
    st = lib.pkv_paged_decode_noalloc(FAKE, FAKE, FAKE, FAKE, _desc(), FAKE, 8, FAKE, huge,
                                      None, 4, 32, -1, 0.1, 512, None, None, None)
    assert st == 3  # PKV_ERR_WORKSPACE


def test_minference_sizes_agree_with_the_oracle():
    """The library's host-side budget arithmetic (how many columns and
    diagonals are kept) against the oracle's, across lengths around the
    caps and the page's default and fixed budgets."""
    import oracle
    for S in (1, 2, 31, 63, 64, 100, 101, 155, 517, 1000, 4096, 20000, 32768, 131072):
        for budget in (0.3, 0.1, 0.05, 0.5, None):
            for vs, ss in ((1000, 6096), (7, 3), (64, 4096)):
                for sink_tokens, recent in ((30, 100), (0, 0), (4, 16)):
                    args = (S, vs, ss, budget, sink_tokens, recent)
                    assert pkv.minference_sizes(*args) == oracle.minference_sizes(*args), args


def test_binding_calls_pass_as_many_arguments_as_the_header_declares():
    """Every pkv_* call in the binding's source passes one argument per
    parameter of its prototype (ctypes would raise only at call time)."""
    import ast
    nparams = {name: len(params) for name, _, params in _prototypes()}
    path = os.path.join(ROOT, "paged_kv_cache_attention_gb300", "__init__.py")
    seen = set()
    for node in ast.walk(ast.parse(open(path).read())):
        if (isinstance(node, ast.Call) and isinstance(node.func, ast.Attribute) and
                node.func.attr in nparams):
            assert not node.keywords and not any(isinstance(a, ast.Starred) for a in node.args)
            assert len(node.args) == nparams[node.func.attr], \
                f"line {node.lineno}: {node.func.attr} takes {nparams[node.func.attr]} arguments"
            seen.add(node.func.attr)
    # every entry point the binding wraps is called through its own name
    assert {"pkv_reshape_and_cache", "pkv_paged_decode", "pkv_paged_decode_noalloc",
            "pkv_varlen_prefill", "pkv_varlen_prefill_contiguous", "pkv_rope_cos_sin_table",
            "pkv_rope_reshape_and_cache", "pkv_minference_sizes",
            "pkv_minference_prefill"} <= seen
