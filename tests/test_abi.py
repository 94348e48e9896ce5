"""Host-side checks of the C ABI: the library builds and loads, exports every
symbol include/relation.h declares, and rejects bad arguments before touching
the GPU (so these run without one)."""
import ctypes
import subprocess

import pytest

from relation_token_mixing_gb300 import binding as rb
from relation_token_mixing_gb300 import build as rbuild

A = 0x10000  # fake, 16-byte aligned addresses: validation fails before any use


@pytest.fixture(scope="module")
def lib():
    return rb.load()


def test_library_exports_every_declared_symbol(lib):
    declared = rb.declared_symbols()
    assert "relation_fwd" in declared and "relation_bwd" in declared
    out = subprocess.run(["nm", "-D", "--defined-only", rbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    for s in declared:
        getattr(lib, s)


def test_version_and_status_strings(lib):
    assert rb.relation_abi_version() == 2
    for code in range(8):
        assert rb.relation_status_string(code) != "unknown status"
    assert rb.relation_status_string(99) == "unknown status"


def _prob(**kw):
    base = dict(B=2, H=3, T=100, d_h=64, dtype=rb.RELATION_BF16, tau_S=1.0, lam=0.5, causal=1,
                layout=rb.RELATION_LAYOUT_BHTD)
    base.update(kw)
    return rb.Problem(base["B"], base["H"], base["T"], base["d_h"], base["dtype"], base["tau_S"], base["lam"],
                      base["causal"], base["layout"])


def _fwd(lib, prob, P1=A, P2=2 * A, V=3 * A, Y=4 * A, L=5 * A):
    return lib.relation_fwd(ctypes.byref(prob), P1, P2, V, Y, L, None)


@pytest.mark.parametrize("kw", [dict(B=0), dict(H=-1), dict(T=0), dict(tau_S=0.0), dict(tau_S=-1.0),
                                dict(tau_S=float("inf")), dict(lam=float("nan")), dict(dtype=7), dict(layout=2),
                                dict(layout=-1)])
def test_invalid_problem_rejected(lib, kw):
    assert _fwd(lib, _prob(**kw)) == 1


@pytest.mark.parametrize("d", [16, 32, 50, 96, 256])
def test_unsupported_head_width(lib, d):
    assert _fwd(lib, _prob(d_h=d)) == 2
    assert rb.relation_bwd_workspace_bytes(_prob(d_h=d)) == 0


@pytest.mark.parametrize("layout", [rb.RELATION_LAYOUT_BHTD, rb.RELATION_LAYOUT_BTHD])
@pytest.mark.parametrize("d,acc", [(48, 64), (60, 64), (64, 64), (80, 128), (128, 128)])
def test_workspace_for_every_width(lib, d, acc, layout):
    """bf16 workspace: the per-query constants of the tensor-core kernels, the fp32 dP1 accumulator
    padded to the tensor-core tile width and, for
    d_h = 60 (rows TMA cannot step through), zero-padded bf16 copies of P1, P2, V, dY."""
    rows = 2 * 3 * 100
    need = rb.relation_bwd_workspace_bytes(_prob(d_h=d, layout=layout))
    pads = 4 * rows * 64 * 2 if d == 60 else 0
    # per-query constants: two floats per query, each head padded to a multiple of 128 queries
    consts = 2 * 3 * 128 * 2 * 4
    assert need >= consts + rows * acc * 4 + pads
    assert need <= consts + rows * acc * 4 + pads + 6 * 256


def test_problem_struct_matches_header():
    """The ctypes mirror has the header's field order and size (ABI 2 added `layout`)."""
    names = [f[0] for f in rb.Problem._fields_]
    assert names == ["B", "H", "T", "d_h", "dtype", "tau_S", "lam", "causal", "layout"]
    assert ctypes.sizeof(rb.Problem) == 4 * 8 + 5 * 4 + 4  # 52 bytes of fields, padded to 8


def test_null_and_misaligned_pointers(lib):
    p = _prob()
    assert _fwd(lib, p, P1=None) == 1
    assert _fwd(lib, p, Y=None) == 1
    assert _fwd(lib, p, V=3 * A + 8) == 3


def test_overlapping_output_rejected(lib):
    p = _prob(B=1, H=1, T=128, d_h=64)
    nbytes = 128 * 64 * 2
    assert _fwd(lib, p, P1=A, P2=A + nbytes, V=A + 2 * nbytes, Y=A + nbytes // 2) == 1
    assert _fwd(lib, p, Y=8 * A, L=8 * A + 16) == 1


def test_workspace_size_and_backward_checks(lib):
    p = _prob(B=2, H=3, T=100, d_h=64)
    need = rb.relation_bwd_workspace_bytes(p)
    rows = 2 * 3 * 100
    assert need >= 2 * 3 * 128 * 8 + rows * 64 * 4  # per-query constants plus the fp32 dP1 accumulator
    pf = _prob(B=2, H=3, T=100, d_h=64, dtype=rb.RELATION_F32)
    assert rb.relation_bwd_workspace_bytes(pf) >= rows * 4
    args = [A * k for k in range(1, 11)]  # P1 P2 V Y L dY dP1 dP2 dV dlambda
    ws = 64 * A
    for name in ("relation_bwd", "relation_bwd_prepare", "relation_bwd_main", "relation_bwd_finish"):
        fn = getattr(lib, name)
        assert fn(ctypes.byref(p), *args, ws, need - 4, None) == 4
        assert fn(ctypes.byref(p), *args[:6], args[0], *args[7:], ws, need, None) == 1  # dP1 aliases P1
        bad = list(args)
        bad[7] += 4
        assert fn(ctypes.byref(p), *bad, ws, need, None) == 3
        assert fn(ctypes.byref(p), *args, None, need, None) == 1


def test_forward_workspace_size_and_checks(lib):
    """relation_fwd_ws: only bf16 d_h = 60 needs a workspace (three zero-padded [rows, 64] bf16
    copies); every call below fails its argument checks before any device call."""
    rows = 2 * 3 * 100
    p = _prob(d_h=60)
    need = rb.relation_fwd_workspace_bytes(p)
    assert need == 3 * ((rows * 64 * 2 + 255) // 256 * 256)
    assert rb.relation_fwd_workspace_bytes(_prob(d_h=60, layout=rb.RELATION_LAYOUT_BTHD)) == need
    for kw in (dict(d_h=48), dict(d_h=64), dict(d_h=80), dict(d_h=128), dict(d_h=60, dtype=rb.RELATION_F32),
               dict(d_h=60, T=0), dict(d_h=50)):
        assert rb.relation_fwd_workspace_bytes(_prob(**kw)) == 0
    M = 1 << 20  # fake, 16-byte aligned addresses 1 MiB apart (each tensor here is 72,000 bytes)
    P1, P2, V, Y, L, ws = M, 2 * M, 3 * M, 4 * M, 5 * M, 8 * M

    def call(prob, ws=ws, nbytes=need, **kw):
        a = dict(P1=P1, P2=P2, V=V, Y=Y, L=L)
        a.update(kw)
        return lib.relation_fwd_ws(ctypes.byref(prob), a["P1"], a["P2"], a["V"], a["Y"], a["L"], ws, nbytes, None)

    assert call(p, ws=None) == 1                 # needed but missing
    assert call(p, ws=ws + 8) == 3               # misaligned
    assert call(p, ws=P1 + 4096) == 1            # overlaps an input
    assert call(p, ws=Y - 16) == 1               # overlaps the output
    assert call(p, ws=L - need + 16) == 1        # overlaps L
    assert call(p, nbytes=need - 16) == 4        # too small
    assert call(p, Y=None) == 1
    assert call(p, V=V + 8) == 3
    assert call(_prob(d_h=60, tau_S=0.0)) == 1
    assert call(_prob(d_h=50)) == 2


@pytest.mark.parametrize("d,dtype,layout,chunk", [
    (64, "bf16", "bhtd", 256), (48, "bf16", "bhtd", 256), (80, "bf16", "bhtd", 128), (128, "bf16", "bhtd", 128),
    (60, "bf16", "bhtd", 512), (64, "bf16", "bthd", 512), (64, "f32", "bhtd", 128), (60, "f32", "bhtd", 128),
    (128, "f32", "bhtd", 64), (128, "f32", "bthd", 512)])
def test_decode_workspace_follows_the_chunk_of_its_path(d, dtype, layout, chunk):
    """Chunk partials (m, l, o[d]) per head and chunk: chunks of 256/128/64 keys (both tensors' rows within
    64 KB) on the bulk-copy path ([B, H, T, d], rows a multiple of 16 bytes), 512 keys otherwise."""
    B, H, T = 2, 3, 1000
    p = _prob(B=B, H=H, T=T, d_h=d, dtype=rb.RELATION_BF16 if dtype == "bf16" else rb.RELATION_F32,
              layout=rb.RELATION_LAYOUT_BHTD if layout == "bhtd" else rb.RELATION_LAYOUT_BTHD)
    assert rb.relation_decode_workspace_bytes(p) == B * H * ((T + chunk - 1) // chunk) * (d + 2) * 4


def test_size_bounds_of_every_entry_point():
    """B*H at most 2^31 - 1 (heads index gridDim.x) and B*H*T at most 2^33 rows (one-dimensional
    grids over rows stay in range); both far beyond what one GPU holds."""
    ws = rb.relation_bwd_workspace_bytes
    assert ws(_prob(B=2 ** 16, H=2 ** 15, T=1, d_h=48)) == 0          # B*H = 2^31
    assert ws(_prob(B=2 ** 16, H=2 ** 15 - 1, T=1, d_h=48)) > 0
    assert ws(_prob(B=2 ** 6, H=2 ** 10, T=2 ** 17 + 1, d_h=48)) == 0   # 2^33 + 2^16 rows
    assert ws(_prob(B=2 ** 6, H=2 ** 10, T=2 ** 17, d_h=48)) > 0        # exactly 2^33 rows
    assert rb.relation_decode_workspace_bytes(_prob(B=2 ** 16, H=2 ** 15, T=1, d_h=48)) == 0


def test_launch_grid_limits_are_refused_before_any_launch(lib):
    """The tensor-core forward holds pairs of 128-row query tiles in gridDim.y (at most 65535), so
    T <= 16,776,960; the CUDA-core (fp32) path holds the heads there, so B*H <= 65535.  Beyond:
    RELATION_ERR_UNSUPPORTED and a workspace size of 0.  At the limit the calls go on to pointer
    validation, which the fake, overlapping addresses here fail (status 1)."""
    t_max = 65535 * 256
    assert _fwd(lib, _prob(B=1, H=1, T=t_max + 1)) == 2
    assert _fwd(lib, _prob(B=1, H=1, T=t_max)) == 1
    assert rb.relation_fwd_workspace_bytes(_prob(B=1, H=1, T=t_max + 1, d_h=60)) == 0
    assert rb.relation_fwd_workspace_bytes(_prob(B=1, H=1, T=t_max, d_h=60)) > 0
    # the backward's tensor-core grid is one-dimensional: the same length is fine there
    assert rb.relation_bwd_workspace_bytes(_prob(B=1, H=1, T=t_max + 1)) > 0
    f32 = rb.RELATION_F32
    for B, H in ((65536, 1), (256, 257)):
        assert _fwd(lib, _prob(B=B, H=H, T=1, dtype=f32)) == 2
        assert rb.relation_bwd_workspace_bytes(_prob(B=B, H=H, T=1, dtype=f32)) == 0
        assert rb.relation_bwd_workspace_bytes(_prob(B=B, H=H, T=1)) > 0   # bf16: tensor-core path
    assert _fwd(lib, _prob(B=65535, H=1, T=1, dtype=f32)) == 1
    assert rb.relation_bwd_workspace_bytes(_prob(B=65535, H=1, T=1, dtype=f32)) > 0


@pytest.mark.parametrize("d,dtype,layout,chunk", [
    (64, "bf16", "bhtd", 256), (48, "bf16", "bhtd", 256), (80, "bf16", "bhtd", 128), (128, "bf16", "bhtd", 128),
    (60, "bf16", "bhtd", 512), (64, "bf16", "bthd", 512), (64, "f32", "bhtd", 128), (48, "f32", "bhtd", 128),
    (60, "f32", "bhtd", 128), (80, "f32", "bhtd", 64), (128, "f32", "bhtd", 64), (128, "f32", "bthd", 512)])
def test_decode_capacity_limit(lib, d, dtype, layout, chunk):
    """Decoding reads a cache of capacity T in at most 8192 chunks (the merge keeps one float per
    chunk in shared memory); a larger capacity is refused with RELATION_ERR_UNSUPPORTED before
    anything is enqueued, and its workspace size is 0."""
    kw = dict(B=1, H=2, d_h=d, dtype=rb.RELATION_BF16 if dtype == "bf16" else rb.RELATION_F32,
              layout=rb.RELATION_LAYOUT_BHTD if layout == "bhtd" else rb.RELATION_LAYOUT_BTHD)
    cap = 8192 * chunk
    assert rb.relation_decode_workspace_bytes(_prob(T=cap, **kw)) == 2 * 8192 * (d + 2) * 4
    assert rb.relation_decode_workspace_bytes(_prob(T=cap + 1, **kw)) == 0
    p = _prob(T=cap + 1, **kw)
    assert lib.relation_decode(ctypes.byref(p), A, 2 * A, 3 * A, 4 * A, 5 * A, 6 * A, 0, 7 * A, None, 8 * A,
                               1 << 30, None) == 2


def test_wait_selftest_limit_is_checked(lib):
    """Limits outside 1..10000 ms are rejected before any device call."""
    for ms in (0, 10001, 2 ** 31):
        assert lib.relation_selftest_wait_timeout(ms, None) == 1


def _lfwd(lib, prob, P1=A, P2=2 * A, I=3 * A, G=4 * A, Y=8 * A, state=None, ws=16 * A):
    return lib.relation_linear_fwd(ctypes.byref(prob), P1, P2, I, G, Y, state, ws, 1 << 30, None)


def _lbwd(lib, prob, ptrs=None, ws=32 * A):
    p = ptrs or [A, 2 * A, 3 * A, 4 * A, 6 * A, 8 * A, 10 * A, 12 * A, 14 * A]  # P1 P2 I G dY dP1 dP2 dI dG
    return lib.relation_linear_bwd(ctypes.byref(prob), *p, 0, ws, 1 << 30, None)


def test_linear_relation_argument_checks(lib):
    """Linear Relation: bf16 only, d_h in {48, 60, 64}; bad problems, NULL, misaligned and
    overlapping pointers are refused before the GPU is touched (every call here fails
    validation: the addresses are fake and nothing may launch)."""
    small = dict(B=1, H=1, T=16, d_h=64)
    assert _lfwd(lib, _prob(**small, dtype=rb.RELATION_F32)) == 2
    assert _lfwd(lib, _prob(B=1, H=1, T=16, d_h=80)) == 2
    assert _lfwd(lib, _prob(B=1, H=1, T=16, d_h=128)) == 2
    assert _lfwd(lib, _prob(**small, tau_S=0.0)) == 1
    assert _lfwd(lib, _prob(**small), P1=None) == 1
    assert _lfwd(lib, _prob(**small), ws=None) == 1
    assert _lfwd(lib, _prob(**small), G=4 * A + 4) == 3
    assert _lfwd(lib, _prob(**small), Y=A + 64) == 1          # Y overlaps P1
    assert _lfwd(lib, _prob(**small), state=4 * A + 64) == 1  # state overlaps G
    assert _lbwd(lib, _prob(**small, dtype=rb.RELATION_F32)) == 2
    bad = [A, 2 * A, 3 * A, 4 * A, 6 * A, 8 * A, 10 * A, 12 * A, 8 * A]  # dG aliases dP1
    assert _lbwd(lib, _prob(**small), bad) == 1
    bad = [A, 2 * A, 3 * A, 4 * A, 6 * A, 8 * A + 8, 10 * A, 12 * A, 14 * A]
    assert _lbwd(lib, _prob(**small), bad) == 3
    assert _lbwd(lib, _prob(**small), ws=None) == 1


def test_prologue_argument_checks(lib):
    """Every call here is refused by validation (the addresses are fake; nothing may launch)."""
    p = _prob(B=1, H=4, T=16, d_h=64)
    f = lib.relation_prologue_fwd
    assert f(ctypes.byref(_prob(B=1, H=3, T=16, d_h=64)), A, 2 * A, 3 * A, 4 * A, 0, 1e4, None, 8 * A, 9 * A, 10 * A,
             None) == 1  # odd H: no head pairs
    assert f(ctypes.byref(p), A, 2 * A, 3 * A, 4 * A, 2, 1e4, None, 8 * A, 9 * A, 10 * A, None) == 1  # pairing 2
    assert f(ctypes.byref(p), A, 2 * A, 3 * A, None, 0, 1e4, None, 8 * A, 9 * A, 10 * A, None) == 1  # no theta
    assert f(ctypes.byref(p), A, 2 * A, 3 * A + 8, 4 * A, 0, 1e4, None, 8 * A, 9 * A, 10 * A, None) == 3
    assert f(ctypes.byref(p), A, 2 * A, 3 * A, 4 * A, 0, 1e4, None, A + 32, 9 * A, 10 * A, None) == 1  # P1 out over X1


def test_step_host_sizes_and_checks(lib):
    """relation_step_host: two slots of one slice's tensors (8 of them), L and backward workspace,
    so the device buffer shrinks with more slices; chunks that do not divide B are refused, and
    every call below fails its argument checks before any device call."""
    p = _prob(B=4, H=2, T=100, d_h=64)
    need = {c: rb.relation_step_host_device_bytes(p, c) for c in (1, 2, 4)}
    for c, n in need.items():
        ps = _prob(B=4 // c, H=2, T=100, d_h=64)
        tb = (4 // c) * 2 * 100 * 64 * 2
        assert n >= 2 * (8 * tb + (4 // c) * 2 * 100 * 4 + rb.relation_bwd_workspace_bytes(ps))
    assert need[4] < need[2] < need[1]
    assert rb.relation_step_host_device_bytes(p, 3) == 0
    assert rb.relation_step_host_device_bytes(p, 0) == 0
    host = [A * k for k in range(1, 11)]  # P1 P2 V dY Y L dP1 dP2 dV dlambda
    buf = 64 * A
    fn = lib.relation_step_host
    assert fn(ctypes.byref(p), *host, 3, buf, need[1], None) == 1  # 3 does not divide B
    assert fn(ctypes.byref(p), None, *host[1:], 1, buf, need[1], None) == 1
    assert fn(ctypes.byref(p), *host, 1, None, need[1], None) == 1
    assert fn(ctypes.byref(p), *host, 1, buf + 4, need[1], None) == 3
    assert fn(ctypes.byref(p), *host, 2, buf, need[2] - 1, None) == 4


def _declarations():
    """(name, return type, parameter types) of every prototype in include/relation.h."""
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "relation.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = []
    for m in re.finditer(r"^\s*((?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?)\s*(relation_[a-z0-9_]+)\s*\(([^)]*)\)\s*;",
                         text, re.M):
        body = m.group(3).strip()
        params = [] if body in ("", "void") else [p.strip() for p in body.split(",")]
        # drop the parameter name (the last identifier after the type), keep the type
        types = [re.sub(r"\s*\b[A-Za-z_][A-Za-z0-9_]*$", "", p) if re.search(r"[\s*]\w+$", p) else p
                 for p in params]
        out.append((m.group(2), m.group(1).replace(" ", ""), types))
    return out


def _ctype_matches(c_type: str, ct) -> bool:
    if "*" in c_type:
        return ct is ctypes.c_void_p or ct is ctypes.c_char_p or hasattr(ct, "_type_") and issubclass(ct, ctypes._Pointer)
    scalar = {"size_t": ctypes.c_size_t, "int": ctypes.c_int, "uint32_t": ctypes.c_uint32, "float": ctypes.c_float,
              "double": ctypes.c_double, "relation_status_t": ctypes.c_int}
    want = scalar.get(c_type.replace("const", "").strip())
    return want is not None and ctypes.sizeof(ct) == ctypes.sizeof(want) and (
        issubclass(ct, (ctypes.c_float, ctypes.c_double)) == issubclass(want, (ctypes.c_float, ctypes.c_double)))


def test_binding_signatures_match_the_header(lib):
    """Every entry point's ctypes argument list matches its prototype, position by position (a pointer where
    the header has a pointer, an integer or float of the header's width elsewhere), and the return type's width
    matches: a slip in the marshalling would otherwise pass wrong arguments silently."""
    decls = _declarations()
    assert len(decls) == len(rb.declared_symbols())
    for name, ret, types in decls:
        f = getattr(lib, name)
        assert f.argtypes is not None, name
        assert len(f.argtypes) == len(types), (name, len(f.argtypes), len(types))
        for k, (c_type, ct) in enumerate(zip(types, f.argtypes)):
            assert _ctype_matches(c_type, ct), (name, k, c_type, ct)
        if ret == "constchar*":
            assert f.restype is ctypes.c_char_p, name
        else:
            assert _ctype_matches(ret, f.restype), (name, ret, f.restype)


def test_binding_constants_match_the_header():
    """Status codes, dtype and layout values and the ABI version in binding.py are the header's."""
    import os
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "relation.h")
    text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
    enum = {n: int(v) for n, v in re.findall(r"\b(RELATION_[A-Z0-9_]+)\s*=\s*(\d+)", text)}
    status = {v: n for n, v in enum.items() if n == "RELATION_OK" or n.startswith("RELATION_ERR_")}
    assert rb.STATUS == status
    for name in ("RELATION_F32", "RELATION_BF16", "RELATION_LAYOUT_BHTD", "RELATION_LAYOUT_BTHD"):
        assert getattr(rb, name) == enum[name], name
    version = int(re.search(r"#define RELATION_ABI_VERSION (\d+)", text).group(1))
    assert rb.relation_abi_version() == version
