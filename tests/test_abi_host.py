"""Host-side tests of the C ABI (no GPU needed).

The library must build, load and export every entry point include/gdn.h
declares; argument validation must reject bad requests with the documented
status before anything is launched.  Device pointers passed here are never
dereferenced: every call below fails validation first.
"""
import ctypes
import os
import re

import pytest

import varlen_gated_delta_gb300 as gdn
from varlen_gated_delta_gb300 import build as gdn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    gdn_build.build()
    return gdn.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_layer_calls():
    names = _declared_functions()
    for n in ("gdn_conv1d_varlen", "gdn_prepare", "gdn_delta_varlen", "gdn_layer_varlen",
              "gdn_workspace_bytes", "gdn_last_error", "gdn_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in gdn.h but not exported"


def test_only_declared_symbols_are_exported():
    """The library hides its internals (-fvisibility=hidden)."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("gdn_")}
    assert ours == set(_declared_functions())


def test_version(lib):
    m = re.search(r"#define GDN_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.gdn_version() == int(m.group(1))


FAKE = ctypes.c_void_p(4096)   # never dereferenced: validation fails first


def _layer(lib, **kw):
    args = dict(qkv=FAKE, w=FAKE, bias=None, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE,
                offsets=FAKE, offsets_host=None, conv_init=FAKE, conv_fin=FAKE,
                state_init=FAKE, out=FAKE, state_fin=FAKE, B=2, N=16, H=4, HQ=2, K=16, V=16,
                Kc=4, D=1, act=1, scale=0.0, dtype=0, ws=FAKE, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    return lib.gdn_layer_varlen(*args.values())


def test_layer_rejects_bad_geometry(lib):
    assert _layer(lib, K=257) == 2
    assert _layer(lib, H=3, HQ=2) == 2
    assert _layer(lib, B=0) == 2
    assert _layer(lib, N=-1) == 2
    assert _layer(lib, Kc=0) == 2
    assert _layer(lib, D=0) == 2
    assert _layer(lib, dtype=7) == 5
    assert _layer(lib, act=3) == 5
    assert _layer(lib, scale=float("nan")) == 2
    assert b"256" in lib.gdn_last_error() or lib.gdn_last_error()


def test_layer_rejects_null_and_workspace(lib):
    assert _layer(lib, qkv=None) == 1
    assert _layer(lib, state_fin=None) == 1
    assert _layer(lib, ws=None) == 8
    assert _layer(lib, ws=ctypes.c_void_p(4096 + 16)) == 8    # misaligned
    assert _layer(lib, ws_bytes=16) == 8


def test_layer_rejects_malformed_host_offsets(lib):
    for bad in ([0, 5, 15], [1, 5, 16], [0, 9, 5, 16]):
        B = len(bad) - 1
        arr = (ctypes.c_int32 * len(bad))(*bad)
        assert _layer(lib, B=B, offsets_host=ctypes.cast(arr, ctypes.c_void_p)) == 4
        assert b"offsets" in lib.gdn_last_error()


def test_overflow_is_reported(lib):
    assert _layer(lib, B=1 << 20, H=64, HQ=64, K=128, V=256) == 3
    assert lib.gdn_conv1d_varlen(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 1 << 20,
                                 1 << 12, 1, 0, None) in (3, 5)


def test_conv_and_delta_validation(lib):
    assert lib.gdn_conv1d_varlen(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 0, 4, 8, 4, 1, 1, 0,
                                 None) == 2
    assert lib.gdn_conv1d_varlen(FAKE, None, None, FAKE, FAKE, FAKE, FAKE, 1, 4, 8, 4, 1, 1, 0,
                                 None) == 1
    assert lib.gdn_delta_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 4, 2, 300, 8,
                                ctypes.c_float(0.0), 0, None) == 2
    assert lib.gdn_prepare(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 3, 2, 8, 8, 0, None) == 2


def test_workspace_bytes(lib):
    n = lib.gdn_workspace_bytes(2, 16, 4, 2, 16, 16, 4, 1, 0)
    assert n > 0 and n % 256 == 0
    assert lib.gdn_workspace_bytes(2, 16, 3, 2, 16, 16, 4, 1, 0) == 0
    big = lib.gdn_workspace_bytes(8, 32768, 32, 16, 128, 128, 4, 1, 1)
    small = lib.gdn_workspace_bytes(8, 1024, 32, 16, 128, 128, 4, 1, 1)
    assert big > small


def test_chunk_threshold_setting(lib):
    default = lib.gdn_chunk_min_len()
    assert default > 0
    assert lib.gdn_set_chunk_min_len(1000) == 0
    assert lib.gdn_chunk_min_len() == 1000
    assert lib.gdn_set_chunk_min_len(0) == 0
    assert lib.gdn_chunk_min_len() == default


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 8)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_conv1d_varlen(x, torch.zeros(8, 4), None, torch.tensor([0, 4], dtype=torch.int32),
                              torch.zeros(1, 8, 3), Kc=4)


def _declared_param_counts():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(gdn_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_header(lib):
    counts = _declared_param_counts()
    for name, n in counts.items():
        fn = getattr(lib, name)
        if fn.argtypes is not None:
            assert len(fn.argtypes) == n, f"{name}: binding has {len(fn.argtypes)} args, header {n}"
        else:
            assert n == 0, f"{name}: binding declares no argtypes but header has {n} params"


def test_kernel_events_hook_validates_id(lib):
    assert lib.gdn_set_kernel_events(3, None, None) == 2
    assert lib.gdn_set_kernel_events(-1, None, None) == 2
    assert lib.gdn_set_kernel_events(0, None, None) == 0


def _layer_capture(lib, cap=4, counts=FAKE, active=None, conv_updates=FAKE, capsule=FAKE, **kw):
    args = dict(qkv=FAKE, w=FAKE, bias=None, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE,
                offsets=FAKE, offsets_host=None, conv_init=FAKE, conv_fin=FAKE,
                state_init=FAKE, out=FAKE, state_fin=FAKE)
    tail = dict(B=2, N=16, H=4, HQ=2, K=16, V=16, Kc=4, D=1, act=1, scale=0.0, dtype=0,
                ws=FAKE, ws_bytes=1 << 30, stream=None)
    for k, v in kw.items():
        (args if k in args else tail)[k] = v
    return lib.gdn_layer_varlen_capture(*args.values(), cap, counts, active, conv_updates,
                                        capsule, *tail.values())


def test_capture_calls_validate_capacity_counts_and_buffers(lib):
    for cap in (0, -1, 9):
        assert _layer_capture(lib, cap=cap) == 2
        assert b"capacity" in lib.gdn_last_error()
    assert _layer_capture(lib, counts=None) == 1
    assert _layer_capture(lib, conv_updates=None, capsule=None) == 1
    # then the plain call's own checks
    assert _layer_capture(lib, K=257) == 2
    assert _layer_capture(lib, ws=None) == 8
    assert _layer_capture(lib, B=1 << 20, H=64, HQ=64, K=128, V=256) == 3
    # the standalone operators
    conv = lambda cap, counts, upd: lib.gdn_conv1d_varlen_capture(
        FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, cap, counts, upd, 2, 16, 8, 4, 1, 1, 0, None)
    assert conv(9, FAKE, FAKE) == 2
    assert conv(2, None, FAKE) == 1
    assert conv(2, FAKE, None) == 1
    delta = lambda cap, counts, capsule: lib.gdn_delta_varlen_capture(
        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, cap, counts, None, capsule, 2, 16, 4, 2, 16,
        16, 0.0, 0, None)
    assert delta(0, FAKE, FAKE) == 2
    assert delta(2, None, FAKE) == 1
    assert delta(2, FAKE, None) == 1


def test_option_calls_validate_option_bits_and_needed_inputs(lib):
    def layer_ex(opts, a=FAKE, b=FAKE, A_log=FAKE, dt_bias=FAKE):
        return lib.gdn_layer_varlen_ex(FAKE, FAKE, None, a, b, A_log, dt_bias, FAKE, None, FAKE,
                                       FAKE, FAKE, FAKE, FAKE, opts, 0, None, None, None, None,
                                       2, 16, 4, 2, 16, 16, 4, 1, 1, 0.0, 0, FAKE, 1 << 30, None)
    assert layer_ex(64) == 5 and b"option" in lib.gdn_last_error()
    assert layer_ex(0, a=None) == 1
    assert layer_ex(0, b=None) == 1
    assert layer_ex(0, A_log=None) == 1
    assert layer_ex(gdn.GDN_OPT_GATE_EXP, b=None) == 1          # the exp gate still needs a and b
    assert layer_ex(gdn.GDN_OPT_NO_DECAY, b=None) == 1
    assert layer_ex(gdn.GDN_OPT_NO_BETA, a=None) == 1
    assert lib.gdn_prepare_ex(FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, 2, 16, 16, 0, 0,
                              None) == 1
    assert lib.gdn_prepare_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, 2, 16, 16, 128, 0,
                              None) == 5
    assert lib.gdn_delta_varlen_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 16, 4, 2, 16, 16,
                                   0.0, 99, 0, None) == 5


def test_dense_call_validation(lib):
    dense = lambda B=2, S=4, H=2, n=16, perch=0, q=FAKE: lib.gdn_gated_delta_dense(
        q, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, B, S, H, n, perch, 0.0, 0, None)
    assert dense(n=257) == 2
    assert dense(n=0) == 2
    assert dense(B=0) == 2
    assert dense(perch=2) == 2
    assert dense(q=None) == 1
    assert dense(B=1 << 16, S=1 << 10, H=64, n=128) == 3
