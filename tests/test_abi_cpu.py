"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/lla.h declares, answers its host-side queries, and rejects bad
arguments before enqueueing anything."""

import ctypes
import os
import re

import pytest

from log_linear_attention_chunkwise_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from log_linear_attention_chunkwise_gb300 import build
        build.build()
    return binding.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "lla.h")).read()
    return sorted(set(re.findall(r"\b(lla_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(binding.SIGNATURES), "binding and header disagree"


def test_status_strings_and_version(lib):
    for code, name in binding.STATUS.items():
        assert lib.lla_status_string(code).decode() == name
    assert lib.lla_version() >= 100


def test_num_levels(lib):
    assert [lib.lla_num_levels(T) for T in (1, 2, 3, 256, 2048, 8192, 32768, 65536)] == \
        [1, 2, 3, 9, 12, 14, 16, 17]
    assert lib.lla_num_levels(0) == 0


def test_workspace_queries(lib):
    n = lib.lla_fwd_workspace_bytes(1, 16, 32768, 128, 128, 64, binding.LLA_BF16)
    assert n > 0 and n % 256 == 0
    assert lib.lla_fwd_workspace_bytes(1, 16, 32768, 128, 128, 48, binding.LLA_BF16) == 0
    assert lib.lla_fwd_workspace_bytes(0, 16, 32768, 128, 128, 64, binding.LLA_BF16) == 0
    assert lib.lla_decode_state_bytes(64, 16, 128, 128, 17) == 64 * 16 * 17 * 128 * 128 * 4
    assert lib.lla_prefill_workspace_bytes(1, 16, 1000) >= 16 * 1000 * 4


NULL = None


def fwd(lib, B=1, H=1, T=64, dk=64, dv=64, chunk=64, in_dt=1, out_dt=0, ws_bytes=1 << 30,
        ptr=ctypes.c_void_p(256)):
    p = ptr
    return lib.lla_fwd(p, p, p, p, p, p, B, H, T, dk, dv, chunk, in_dt, out_dt, p, ws_bytes, NULL,
                       NULL)


@pytest.mark.parametrize("kw,code", [
    (dict(chunk=48), 2), (dict(T=100), 2), (dict(dk=96), 2), (dict(dv=8), 2),
    (dict(B=-1), 1), (dict(in_dt=7), 1), (dict(out_dt=9), 1), (dict(in_dt=0, out_dt=1), 2),
    (dict(ws_bytes=0), 3), (dict(ptr=ctypes.c_void_p(0)), 1), (dict(ptr=ctypes.c_void_p(8)), 1),
    (dict(T=1 << 25), 2), (dict(B=70000), 2),
])
def test_fwd_validation_rejects_before_launch(lib, kw, code):
    assert fwd(lib, **kw) == code


def test_fwd_empty_is_a_noop(lib):
    assert fwd(lib, T=0, ptr=ctypes.c_void_p(0), ws_bytes=0) == 0
    assert fwd(lib, B=0, ptr=ctypes.c_void_p(0), ws_bytes=0) == 0


def test_decode_validation(lib):
    p = ctypes.c_void_p(256)
    args = lambda **kw: [kw.get("S", p), p, p, p, p, p, p, p, p, kw.get("B", 2), 2,
                         kw.get("dk", 64), 64, kw.get("Ls", 17), kw.get("dt", 1), NULL, NULL]
    assert lib.lla_decode_step(*args(dk=48)) == 2
    assert lib.lla_decode_step(*args(Ls=0)) == 2
    assert lib.lla_decode_step(*args(Ls=41)) == 2
    assert lib.lla_decode_step(*args(dt=3)) == 1
    assert lib.lla_decode_step(*args(S=ctypes.c_void_p(0))) == 1
    assert lib.lla_decode_step(*args(B=0, S=ctypes.c_void_p(0))) == 0


def test_prefill_validation(lib):
    p = ctypes.c_void_p(256)
    # bit_length(T) must fit in Ls slots
    assert lib.lla_prefill_state(p, p, p, p, p, 1, 1, 8, 64, 64, 3, 1, p, 1 << 20, NULL, NULL) == 2
    assert lib.lla_prefill_state(p, p, p, p, p, 1, 1, 8, 64, 64, 4, 1, p, 0, NULL, NULL) == 3


def test_bwd_validation(lib):
    p = ctypes.c_void_p(256)

    def bwd(B=1, T=256, dk=64, chunk=64, dt=1, ws=1 << 30, ptr=p):
        return lib.lla_bwd(ptr, p, p, p, p, p, p, p, p, p, p, B, 1, T, dk, 64, chunk, dt,
                           p, ws, NULL, NULL)
    assert bwd(chunk=128) == 2          # the backward takes chunks up to 64
    assert bwd(dk=48) == 2
    assert bwd(T=100) == 2
    assert bwd(dt=5) == 1
    assert bwd(ws=0) == 3
    assert bwd(ptr=ctypes.c_void_p(0)) == 1
    assert bwd(B=0, ptr=ctypes.c_void_p(0), ws=0) == 0
    assert lib.lla_bwd_workspace_bytes(1, 1, 256, 64, 64, 128, 1) == 0
    # Fenwick nodes [BH][N][dk][dv] plus block states, both fp32
    assert lib.lla_bwd_workspace_bytes(1, 2, 256, 64, 64, 64, 1) >= 2 * (4 + 4) * 64 * 64 * 4


def test_gdn_validation(lib):
    p = ctypes.c_void_p(256)

    def fwd(B=1, T=64, dk=64, Ls=0, st=NULL, dt=1, q=p, k=p, v=p, out=p, ws=p, wsb=1 << 30):
        return lib.lla_gdn_fwd(q, k, v, p, p, p, out, st, B, 1, T, dk, 64, Ls, dt, ws, wsb, NULL)
    assert fwd(dk=48) == 2
    assert fwd(T=(1 << 24) + 1) == 2
    assert fwd(st=p, Ls=6) == 2          # 64 tokens need bit_length(64) = 7 slots
    assert fwd(dt=4) == 1
    assert fwd(B=0) == 0
    assert fwd(ws=NULL) == 1
    assert fwd(ws=ctypes.c_void_p(256 + 16)) == 1   # workspace not 256-byte aligned
    assert fwd(k=ctypes.c_void_p(256 + 4)) == 1     # k not 16-byte aligned
    assert fwd(out=ctypes.c_void_p(256 + 8)) == 1   # out not 16-byte aligned
    assert fwd(q=ctypes.c_void_p(256 + 2)) == 1     # q, v read in 16-byte pieces
    assert fwd(v=ctypes.c_void_p(256 + 2)) == 1
    assert fwd(wsb=lib.lla_gdn_fwd_workspace_bytes(1, 1, 64, 64, 64) - 1) == 1
    # per chunk of 64: q~^T and w^T [2][dk][64], H [dk][dv], the decay (fp32)
    assert lib.lla_gdn_fwd_workspace_bytes(1, 1, 64, 64, 64) >= (2 * 64 * 64 + 64 * 64 + 1) * 4
    assert lib.lla_gdn_fwd_workspace_bytes(2, 3, 130, 32, 16) >= 2 * 3 * 3 * (2 * 32 * 64 + 32 * 16 + 1) * 4
    assert lib.lla_gdn_fwd_workspace_bytes(0, 3, 130, 32, 16) == 0
    assert lib.lla_gdn_decode_step(p, p, p, p, p, p, p, p, p, 1, 1, 64, 64, 41, 1, NULL, NULL) == 2
    assert lib.lla_gdn_decode_step(NULL, p, p, p, p, p, p, p, p, 1, 1, 64, 64, 17, 1, NULL, NULL) == 1


def test_device_error_check_rejects_null(lib):
    code = ctypes.c_int32(7)
    assert lib.lla_device_error_check(NULL, ctypes.byref(code), NULL) == 1
    assert code.value == 7   # untouched: nothing was read


def test_noalloc_checks_arguments_in_lla_fwd_order(lib):
    """A bad call gets the status lla_fwd would give it, whatever its size:
    shape and pointer errors come before the scratch-size refusal."""
    p = ctypes.c_void_p(256)
    big = dict(B=1, H=16, T=32768)

    def noalloc(ptr=p, chunk=64, B=1, H=1, T=64, d=64, in_dt=1, out_dt=0):
        return lib.lla_fwd_noalloc(ptr, p, p, p, p, p, B, H, T, d, d, chunk, in_dt, out_dt, NULL,
                                   NULL)
    assert noalloc(chunk=48, **big) == 2
    assert noalloc(ptr=ctypes.c_void_p(0), d=128, **big) == 1
    assert noalloc(ptr=ctypes.c_void_p(8), d=128, **big) == 1
    assert noalloc(out_dt=9, d=128, **big) == 1
    assert noalloc(B=0, ptr=ctypes.c_void_p(0)) == 0


def test_fwd_lambda_mlp_validation(lib):
    p = ctypes.c_void_p(256)

    def call(d=p, Dd=64, T=64, dk=64, ws=1 << 30, wsp=p, W1=p):
        return lib.lla_fwd_lambda_mlp(p, p, p, p, d, W1, p, p, p, 1, 1, T, dk, dk, Dd, 64, 1, 0,
                                      wsp, ws, NULL, NULL)
    assert call(Dd=0) == 2
    assert call(Dd=300) == 2
    assert call(dk=48) == 2
    assert call(d=NULL) == 1
    assert call(W1=NULL) == 1
    assert call(d=ctypes.c_void_p(256 + 8)) == 1
    assert call(ws=0) == 3
    assert call(wsp=ctypes.c_void_p(256 + 16)) == 1
    # enough for lambda staged in the workspace plus the forward's own workspace
    n = lib.lla_fwd_lambda_mlp_workspace_bytes(2, 3, 2048, 128, 128, 128, 64, 1)
    assert n >= 2 * 3 * 2048 * 12 * 4 + lib.lla_fwd_workspace_bytes(2, 3, 2048, 128, 128, 64, 1)
    assert lib.lla_fwd_lambda_mlp_workspace_bytes(2, 3, 2048, 128, 128, 0, 64, 1) == 0
