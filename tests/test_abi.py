"""C ABI contract tests (CPU, no GPU): exported symbols, prototypes, host-side errors.

The analogue of the reference's AST contract tests (b12x PR #137, Summary:
"Add AST contract tests so future shared-kernel signature changes fail in unit
tests"): the header is parsed and compared with what the library exports and
with the ctypes prototypes the binding declares.  Calls made here touch no
device: they fail validation, or only compute sizes.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "b4moe.h")


@pytest.fixture(scope="module")
def b4():
    import __graft_entry__

    __graft_entry__._build_module().build()
    import w4a16_moe_gb300 as mod

    return mod


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = {}
    for m in re.finditer(r"\n([A-Za-z_][\w\s\*]*?)(b4_\w+)\s*\(([^;{]*?)\)\s*;", text):
        ret, name, args = m.group(1).strip(), m.group(2), m.group(3)
        nargs = 0 if args.strip() in ("void", "") else len(args.split(","))
        decls[name] = (ret, nargs)
    return decls


def test_header_declares_the_expected_entry_points():
    names = set(_declared())
    assert {"b4_route_capacity_tokens", "b4_workspace_bytes", "b4_prepared_sizes", "b4_prepare_weights",
            "b4_route_pack", "b4_fused_moe", "b4_check_status", "b4_wait_self_test", "b4_status_string",
            "b4_last_error"} <= names


def test_wait_self_test_validates_before_launch(b4):
    """The bounded-wait diagnostic refuses a missing or short status word and
    a limit outside 1 .. 1000000 us before it touches a device."""
    lib = b4.raw_lib()
    assert lib.b4_wait_self_test(None, 0, 1000, None) == b4.B4_ERR_INVALID_ARGUMENT
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    assert lib.b4_wait_self_test(fake, 4, 1000, None) == b4.B4_ERR_INVALID_ARGUMENT
    assert lib.b4_wait_self_test(fake, 8, 0, None) == b4.B4_ERR_INVALID_ARGUMENT
    assert lib.b4_wait_self_test(fake, 8, 1000001, None) == b4.B4_ERR_INVALID_ARGUMENT
    assert "limit_us" in b4.last_error()


def test_library_exports_every_declared_symbol(b4):
    out = subprocess.run(["nm", "-D", "--defined-only", b4.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared():
        assert name in exported, name
        assert getattr(ctypes.CDLL(b4.LIB_PATH), name) is not None


def test_ctypes_prototypes_match_header_arity(b4):
    lib = b4.raw_lib()
    for name, (_, nargs) in _declared().items():
        fn = getattr(lib, name)
        assert len(fn.argtypes) == nargs, (name, len(fn.argtypes), nargs)
    assert set(b4.EXPORTED) == set(_declared())


def test_config_struct_layout_matches_header(b4):
    text = open(HEADER).read()
    body = re.search(r"typedef struct b4_moe_config \{(.*?)\} b4_moe_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"(\w+)\s*;", body)
    assert [f[0] for f in b4._Config._fields_] == fields
    # eight int32, the expert_map pointer, three floats, tail padding to 8 bytes
    assert b4._Config.swiglu_alpha.offset == 40 and b4._Config.swiglu_limit.offset == 48
    assert ctypes.sizeof(b4._Config) == 8 * 4 + 8 + 3 * 4 + 4


def test_activation_enum_matches_header(b4):
    text = open(HEADER).read()
    body = re.search(r"typedef enum b4_activation \{(.*?)\} b4_activation;", text, re.S).group(1)
    values = {k: int(v) for k, v in re.findall(r"B4_ACT_(\w+)\s*=\s*(\d+)", body)}
    assert values == {"SILU_SWIGLU": b4.SILU, "RELU2": b4.RELU2, "SWIGLU_OAI": b4.SWIGLU_OAI}


def _cfg(b4, **kw):
    base = dict(m=4, top_k=2, num_global_experts=8, num_local_experts=8, hidden=256, inter=512)
    base.update(kw)
    return b4.MoEConfig(**base)


def test_capacity_and_workspace_sizes_are_power_of_two_stable(b4):
    assert [b4.route_capacity_tokens(m) for m in (0, 1, 2, 3, 5, 64, 65)] == [1, 1, 2, 4, 8, 64, 128]
    sizes = {m: b4.workspace_bytes(_cfg(b4, m=m), b4.SILU) for m in (33, 40, 64, 65, 128)}
    assert sizes[33] == sizes[40] == sizes[64] < sizes[65] == sizes[128]
    for m in range(0, 300, 7):
        assert b4.workspace_bytes(_cfg(b4, m=m), b4.SILU) <= b4.workspace_bytes(_cfg(b4, m=m + 7), b4.SILU)


def test_clamped_swiglu_shares_the_gated_layout(b4):
    for m in (1, 16, 300):
        assert b4.workspace_bytes(_cfg(b4, m=m), b4.SWIGLU_OAI) == b4.workspace_bytes(_cfg(b4, m=m), b4.SILU)
    for which in (0, 1):
        assert b4.prepared_sizes(_cfg(b4), which, b4.SWIGLU_OAI) == b4.prepared_sizes(_cfg(b4), which, b4.SILU)
    assert b4.prepared_sizes(_cfg(b4), 0, b4.SWIGLU_OAI) != b4.prepared_sizes(_cfg(b4), 0, b4.RELU2)


@pytest.mark.parametrize("kw", [
    dict(swiglu_limit=0.0), dict(swiglu_limit=-7.0), dict(swiglu_limit=float("nan")),
    dict(swiglu_alpha=float("inf")), dict(swiglu_alpha=float("nan")), dict(swiglu_beta=float("-inf")),
])
def test_clamped_swiglu_parameters_are_checked(b4, kw):
    """Checked before anything else happens, so m = 0 (no pointers, no device) reaches the check."""
    lib = b4.raw_lib()
    bad = _cfg(b4, m=0, **kw)._c()
    st = lib.b4_fused_moe(ctypes.byref(bad), *([None] * 9), b4.SWIGLU_OAI, None, None, 0, None)
    assert st == b4.B4_ERR_INVALID_ARGUMENT and "swiglu" in b4.last_error()
    # the other activations ignore the three fields
    assert lib.b4_fused_moe(ctypes.byref(bad), *([None] * 9), b4.SILU, None, None, 0, None) == b4.B4_OK
    good = _cfg(b4, m=0, swiglu_limit=float("inf"))._c()
    assert lib.b4_fused_moe(ctypes.byref(good), *([None] * 9), b4.SWIGLU_OAI, None, None, 0, None) == b4.B4_OK


def test_prepared_sizes(b4):
    cb, sb = b4.prepared_sizes(_cfg(b4), 0, b4.SILU)
    # SwiGLU W13: I=512 -> 8 tiles of 128 rows; H=256 -> 4 stages of 64
    assert cb == 8 * 8 * 4 * 4096 and sb == 8 * 8 * 4 * 512
    cb, sb = b4.prepared_sizes(_cfg(b4, format=b4.MXFP4, hidden=2880, inter=1440), 1, b4.SILU)
    # W2: H=2880 -> 23 tiles; I=1440 -> 23 stages (padded to 1472)
    assert cb == 8 * 23 * 23 * 4096 and sb == 8 * 23 * 23 * 256


@pytest.mark.parametrize("kw,fragment", [
    (dict(top_k=0), "top_k"),
    (dict(m=-1), "m ="),
    (dict(hidden=250), "hidden"),
    (dict(inter=8), "inter"),
    (dict(format=7), "format"),
    (dict(num_global_experts=9), "expert_map"),
    (dict(num_local_experts=0), "num_local_experts"),
    (dict(path=1, m=65), "decode path"),
])
def test_invalid_configs_are_rejected_before_any_launch(b4, kw, fragment):
    with pytest.raises(b4.B4Error) as ei:
        b4.workspace_bytes(_cfg(b4, **kw), b4.SILU)
    assert ei.value.status == b4.B4_ERR_INVALID_ARGUMENT
    assert fragment in str(ei.value)


def test_null_pointers_and_bad_activation_are_rejected(b4):
    lib = b4.raw_lib()
    c = _cfg(b4)._c()
    st = lib.b4_fused_moe(ctypes.byref(c), None, None, None, None, None, None, None, None, None, 0, None, None, 0,
                          None)
    assert st == b4.B4_ERR_INVALID_ARGUMENT and "null" in b4.last_error()
    assert lib.b4_workspace_bytes(ctypes.byref(c), 9) == 0 and "activation" in b4.last_error()
    assert lib.b4_fused_moe(None, *([None] * 9), 0, None, None, 0, None) == b4.B4_ERR_INVALID_ARGUMENT
    # m = 0 is a no-op that needs no pointers and no device
    c0 = _cfg(b4, m=0)._c()
    assert lib.b4_fused_moe(ctypes.byref(c0), *([None] * 9), 0, None, None, 0, None) == b4.B4_OK


def test_status_strings(b4):
    assert [b4.status_string(s) for s in range(6)] == [
        "B4_OK", "B4_ERR_INVALID_ARGUMENT", "B4_ERR_UNSUPPORTED_DEVICE", "B4_ERR_WORKSPACE_TOO_SMALL",
        "B4_ERR_CUDA", "B4_ERR_TIMEOUT"]
    assert b4.status_string(99) == "B4_UNKNOWN_STATUS"


def test_linear_entry_points_validate_on_the_host(b4):
    """b4_linear takes one expert, top-1, no expert_map; sizes need no device."""
    cfg = b4.linear_config(16, 4096, 4096)
    assert b4.linear_workspace_bytes(cfg) > 0
    for kw, fragment in ((dict(top_k=2), "top_k = 1"), (dict(num_local_experts=2, num_global_experts=2), "one expert"),
                         (dict(inter=40), "inter")):
        bad = b4.linear_config(16, 4096, 4096)
        for k_, v in kw.items():
            setattr(bad, k_, v)
        with pytest.raises(b4.B4Error) as ei:
            b4.linear_workspace_bytes(bad)
        assert fragment in str(ei.value)
    lib = b4.raw_lib()
    c = cfg._c()
    assert lib.b4_linear(ctypes.byref(c), None, None, None, None, None, None, 0, None) == b4.B4_ERR_INVALID_ARGUMENT
    assert "null" in b4.last_error()
    c0 = b4.linear_config(0, 4096, 4096)._c()  # m = 0: a no-op
    assert lib.b4_linear(ctypes.byref(c0), None, None, None, None, None, None, 0, None) == b4.B4_OK
    # MXFP4 takes no global scale, NVFP4 needs one (checked before any pointer is used)
    one = ctypes.c_float(1.0)
    cmx = b4.linear_config(2, 256, 256, format=b4.MXFP4)._c()
    buf = ctypes.create_string_buffer(1 << 12)
    p = ctypes.addressof(buf)
    assert lib.b4_linear(ctypes.byref(cmx), p, p, p, ctypes.addressof(one), p, p, 1 << 12,
                         None) == b4.B4_ERR_INVALID_ARGUMENT
    assert "global scale" in b4.last_error()


def test_linear_workspace_is_monotone_and_capacity_stable(b4):
    """One workspace serves every m up to the next power of two, and the
    size never shrinks as m grows (the same contract as b4_workspace_bytes)."""
    for fmt, n, k in ((b4.NVFP4, 4096, 4096), (b4.MXFP4, 1440, 2880), (b4.NVFP4, 256, 8192)):
        sizes = [b4.linear_workspace_bytes(b4.linear_config(m, n, k, format=fmt)) for m in range(0, 300, 5)]
        assert all(a <= b for a, b in zip(sizes, sizes[1:]))
        assert (b4.linear_workspace_bytes(b4.linear_config(33, n, k, format=fmt))
                == b4.linear_workspace_bytes(b4.linear_config(64, n, k, format=fmt)))
