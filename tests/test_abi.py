"""Host-only checks of the C ABI: the library builds, loads, exports every symbol that
include/swa_attn.h declares, and rejects bad arguments before launching anything (these calls
return from the argument checks, so they need no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swa_attn.h")

FAKE = 0x10000  # 16-byte-aligned fake device address; never dereferenced by these calls


@pytest.fixture(scope="module")
def lib():
    import sliding_window_flash_gb300 as swa
    from sliding_window_flash_gb300 import build as swa_build

    if not os.path.exists(swa.library_path()):
        swa_build.build()
    return swa.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(swa_[a-z_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("swa_attn_fwd", "swa_attn_bwd", "swa_attn_bwd_workspace_bytes", "swa_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    import sliding_window_flash_gb300 as swa

    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in swa.SIGNATURES, f"binding has no signature for {name}"


def _declared_statuses():
    """{value: name} of the swa_status enum in include/swa_attn.h."""
    text = open(os.path.join(ROOT, "include", "swa_attn.h")).read()
    return {int(v): n for n, v in re.findall(r"\b(SWA_(?:OK|ERR_[A-Z_]+))\s*=\s*(\d+)", text)}


def test_version_and_strerror(lib):
    import sliding_window_flash_gb300 as swa

    assert lib.swa_version() >= 100
    declared = _declared_statuses()
    assert declared and sorted(declared) == list(range(len(declared)))
    for code, name in declared.items():
        msg = lib.swa_strerror(code)
        assert msg.startswith(name.encode()), (code, msg)
        assert swa.STATUS[code] == name
    assert b"UNKNOWN" in lib.swa_strerror(99)


def _fwd(lib, B=1, Hq=2, Hkv=1, N=16, D=64, W=4, scale=0.125, ptrs=None, f16=False):
    p = ptrs or [FAKE] * 5
    fn = lib.swa_attn_fwd_f16 if f16 else lib.swa_attn_fwd
    return fn(*p, B, Hq, Hkv, N, D, W, scale, None)


def _bwd(lib, B=1, Hq=2, Hkv=1, N=16, D=64, W=4, scale=0.125, ptrs=None, ws=FAKE, ws_bytes=1 << 20,
         f16=False):
    p = ptrs or [FAKE] * 9
    fn = lib.swa_attn_bwd_f16 if f16 else lib.swa_attn_bwd
    return fn(*p, B, Hq, Hkv, N, D, W, scale, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), 1), (dict(B=0), 1), (dict(Hq=0), 1), (dict(Hkv=0), 1), (dict(W=0), 1),
    (dict(W=-3), 1), (dict(Hq=3, Hkv=2), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(D=96), 2), (dict(D=512), 2), (dict(D=32), 2),
])
@pytest.mark.parametrize("f16", [False, True], ids=["bf16", "fp16"])
def test_fwd_rejects_bad_sizes(lib, kw, code, f16):
    assert _fwd(lib, f16=f16, **kw) == code
    assert _bwd(lib, f16=f16, **kw) == code


@pytest.mark.parametrize("f16", [False, True], ids=["bf16", "fp16"])
def test_null_and_misaligned_pointers(lib, f16):
    assert _fwd(lib, ptrs=[FAKE, 0, FAKE, FAKE, FAKE], f16=f16) == 1
    assert _fwd(lib, ptrs=[FAKE, FAKE, FAKE + 8, FAKE, FAKE], f16=f16) == 3
    assert _fwd(lib, ptrs=[FAKE, FAKE, FAKE, FAKE, FAKE + 4], f16=f16) == 3
    assert _bwd(lib, ptrs=[FAKE] * 8 + [0], f16=f16) == 1
    assert _bwd(lib, ptrs=[FAKE] * 8 + [FAKE + 2], f16=f16) == 3
    assert _bwd(lib, ws=0, f16=f16) == 6


def _fwd_ex(lib, B=1, Hq=2, Hkv=1, Lq=16, Lk=40, D=64, W=4, causal=1, scale=0.125, f16=0):
    return lib.swa_attn_fwd_ex(*([FAKE] * 5), B, Hq, Hkv, Lq, Lk, D, W, causal, scale, f16, None)


def _bwd_ex(lib, B=1, Hq=2, Hkv=1, Lq=16, Lk=40, D=64, W=4, causal=1, scale=0.125, f16=0,
            ws_bytes=1 << 20):
    return lib.swa_attn_bwd_ex(*([FAKE] * 9), B, Hq, Hkv, Lq, Lk, D, W, causal, scale, f16, FAKE,
                               ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Lq=41), 1), (dict(Lq=0), 1), (dict(Lk=0), 1), (dict(causal=2), 1), (dict(causal=-1), 1),
    (dict(f16=2), 1), (dict(W=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(D=512), 2),
])
def test_ex_entry_points_reject_bad_arguments(lib, kw, code):
    assert _fwd_ex(lib, **kw) == code
    assert _bwd_ex(lib, **kw) == code


def test_ex_workspace_follows_the_query_length(lib):
    need = lib.swa_attn_bwd_workspace_bytes(1, 2, 16, 64)
    assert _bwd_ex(lib, ws_bytes=need - 1) == 6


def _f32_need(lib, B=1, Hq=2, Hkv=1, Lq=16, Lk=40, D=64):
    return lib.swa_attn_f32_workspace_bytes(B, Hq, Hkv, Lq, Lk, D)


def _fwd_f32(lib, B=1, Hq=2, Hkv=1, Lq=16, Lk=40, D=64, W=4, causal=1, scale=0.125, ws=FAKE,
             ws_bytes=None, ptrs=None):
    ws_bytes = _f32_need(lib) if ws_bytes is None else ws_bytes
    ptrs = [FAKE] * 5 if ptrs is None else ptrs
    return lib.swa_attn_fwd_f32(*ptrs, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, ws, ws_bytes, None)


def _bwd_f32(lib, B=1, Hq=2, Hkv=1, Lq=16, Lk=40, D=64, W=4, causal=1, scale=0.125, ws=FAKE,
             ws_bytes=None, ptrs=None):
    ws_bytes = _f32_need(lib) if ws_bytes is None else ws_bytes
    ptrs = [FAKE] * 9 if ptrs is None else ptrs
    return lib.swa_attn_bwd_f32(*ptrs, B, Hq, Hkv, Lq, Lk, D, W, causal, scale, ws, ws_bytes, None)


def test_f32_workspace_size():
    """Bytes: bf16 copies of q, k, v, a query-shaped slot, dq, dk, dv, fp32 Delta, then the bf16
    residuals of q and k and a second query-shaped slot, each region rounded up to 256 bytes."""
    import sliding_window_flash_gb300 as swa

    lib = swa.load()

    def r(x):
        return (x + 255) // 256 * 256

    B, Hq, Hkv, Lq, Lk, D = 2, 4, 2, 100, 300, 128
    qb, kb = r(B * Hq * Lq * D * 2), r(B * Hkv * Lk * D * 2)
    assert _f32_need(lib, B, Hq, Hkv, Lq, Lk, D) == 5 * qb + 5 * kb + r(B * Hq * Lq * 4)
    assert swa.swa_attn_f32_workspace_bytes(B, Hq, Hkv, Lq, Lk, D) == 5 * qb + 5 * kb + r(
        B * Hq * Lq * 4)
    assert _f32_need(lib, Lq=41) == 0 and _f32_need(lib, D=96) == 0 and _f32_need(lib, B=0) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(Lq=41), 1), (dict(Lq=0), 1), (dict(causal=2), 1), (dict(W=0), 1),
    (dict(Hq=3, Hkv=2), 1), (dict(scale=0.0), 1), (dict(D=512), 2),
    (dict(ws=0), 6), (dict(ws_bytes=0), 6), (dict(ws=FAKE + 8), 3),
])
def test_f32_entry_points_reject_bad_arguments(lib, kw, code):
    assert _fwd_f32(lib, **kw) == code
    assert _bwd_f32(lib, **kw) == code


def test_f32_workspace_too_small_by_one_byte(lib):
    assert _fwd_f32(lib, ws_bytes=_f32_need(lib) - 1) == 6
    assert _bwd_f32(lib, ws_bytes=_f32_need(lib) - 1) == 6


def test_f32_null_and_misaligned_pointers(lib):
    for i in range(5):
        ptrs = [FAKE] * 5
        ptrs[i] = 0
        assert _fwd_f32(lib, ptrs=ptrs) == 1
        ptrs[i] = FAKE + 4
        assert _fwd_f32(lib, ptrs=ptrs) == 3
    for i in range(9):
        ptrs = [FAKE] * 9
        ptrs[i] = 0
        assert _bwd_f32(lib, ptrs=ptrs) == 1
        ptrs[i] = FAKE + 8
        assert _bwd_f32(lib, ptrs=ptrs) == 3


def test_head_dims(lib):
    """D in {64, 128, 256} passes the checks (workspaces are sized), anything else is refused."""
    for D in (64, 128, 256):
        assert lib.swa_attn_bwd_workspace_bytes(1, 2, 100, D) > 0
        assert _f32_need(lib, D=D) > 0
    for D in (32, 96, 192, 512):
        assert lib.swa_attn_bwd_workspace_bytes(1, 2, 100, D) == 0
        assert _fwd_ex(lib, D=D) == 2 and _bwd_ex(lib, D=D) == 2


def _host(lib, B=1, Hq=2, Hkv=1, N=16, D=64, W=4, scale=0.125, U=1, ws=FAKE, ws_bytes=None,
          ptrs=None):
    ws_bytes = lib.swa_attn_host_workspace_bytes(B, Hq, Hkv, N, D, U) if ws_bytes is None \
        else ws_bytes
    ptrs = [FAKE] * 9 if ptrs is None else ptrs
    return lib.swa_attn_fwd_bwd_host(*ptrs, B, Hq, Hkv, N, D, W, scale, U, ws, ws_bytes, None)


def test_host_pipeline_workspace_size(lib):
    """Three slots, each q, dO, o, dq (q-shaped), k, v, dk, dv (k-shaped), lse and Delta for
    min(U, B Hkv) groups, every buffer rounded up to 256 bytes."""
    def r(x):
        return (x + 255) // 256 * 256

    B, Hq, Hkv, N, D = 2, 8, 2, 300, 128
    for U in (1, 3, 4, 9):
        u = min(U, B * Hkv)
        G = Hq // Hkv
        slot = 4 * r(u * G * N * D * 2) + 4 * r(u * N * D * 2) + 2 * r(u * G * N * 4)
        assert lib.swa_attn_host_workspace_bytes(B, Hq, Hkv, N, D, U) == 3 * slot
    assert lib.swa_attn_host_workspace_bytes(B, Hq, Hkv, N, D, 0) == 0
    assert lib.swa_attn_host_workspace_bytes(B, Hq, 3, N, D, 1) == 0
    assert lib.swa_attn_host_workspace_bytes(B, Hq, Hkv, N, 96, 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(U=0, ws_bytes=1 << 20), 1), (dict(W=0), 1), (dict(N=0, ws_bytes=1 << 20), 1),
    (dict(Hq=3, Hkv=2, ws_bytes=1 << 20), 1), (dict(D=512, ws_bytes=1 << 20), 2),
    (dict(ws=0), 6), (dict(ws_bytes=0), 6), (dict(ws=FAKE + 8), 3),
])
def test_host_pipeline_rejects_bad_arguments(lib, kw, code):
    assert _host(lib, **kw) == code


def test_host_pipeline_null_and_misaligned(lib):
    for i in range(9):
        ptrs = [FAKE] * 9
        ptrs[i] = 0
        assert _host(lib, ptrs=ptrs) == 1
        ptrs[i] = FAKE + 4
        assert _host(lib, ptrs=ptrs) == 3
    need3 = lib.swa_attn_host_workspace_bytes(1, 2, 1, 16, 64, 1)
    assert _host(lib, ws_bytes=need3 * 2 // 3 - 1) == 6  # below two slots


def test_workspace_checks(lib):
    need = lib.swa_attn_bwd_workspace_bytes(2, 4, 100, 128)
    assert need == ((2 * 4 * 100 * 4 + 255) // 256) * 256
    assert lib.swa_attn_bwd_workspace_bytes(0, 4, 100, 128) == 0
    assert lib.swa_attn_bwd_workspace_bytes(1, 4, 100, 80) == 0
    assert _bwd(lib, ws=0) == 6
    assert _bwd(lib, ws_bytes=lib.swa_attn_bwd_workspace_bytes(1, 2, 16, 64) - 1) == 6
    assert _bwd(lib, ws=FAKE + 8) == 3


def test_index_range_limits(lib):
    # B*Hq*N rows must stay below 2^31.
    assert _fwd(lib, B=1 << 12, Hq=1 << 10, Hkv=1, N=1 << 10) == 1


def test_python_binding_refuses_cpu_tensors():
    import torch

    import sliding_window_flash_gb300 as swa

    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        swa.swa_attn_fwd(q, k, k, 4)
    with pytest.raises(ValueError):
        swa.swa_attn_fwd(q.half(), k.half(), k.half(), 4)
    with pytest.raises(ValueError):
        swa.swa_attn_fwd(q.float(), k.float(), k.float(), 4)
    with pytest.raises(TypeError):
        swa.swa_attn_fwd(q.double(), k.double(), k.double(), 4)
