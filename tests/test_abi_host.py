"""The C ABI library loads, exports every symbol include/pa.h declares, and
refuses bad arguments on the host before any CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

from invariant_paged_kv_gb300 import build, pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pa.load()


def declared_functions(header="pa.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pa_write_kv", "pa_attention", "pa_attention_workspace_bytes",
                 "pa_read_status", "pa_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # the binding wraps exactly the declared boundary
    assert set(declared_functions()) == set(pa.EXPORTS)
    # and the test hooks of the separate header
    for name in declared_functions("pa_test.h"):
        assert hasattr(lib, name), name
    assert set(declared_functions("pa_test.h")) == set(pa.TEST_EXPORTS)


def test_status_strings(lib):
    for code, name in pa.STATUS_NAMES.items():
        assert lib.pa_status_string(code).decode() == name


def test_split_tokens(lib):
    assert lib.pa_split_tokens() == 512


def test_workspace_bytes_host_only(lib):
    f = lib.pa_attention_workspace_bytes
    # decode-only bf16, H32/Hkv8/D128/bs16, 64 lanes, ctx <= 16384, total 205000
    n = f(64, 64, 1, 16384, 205000, 32, 8, 128, 16, 1)
    pairs = 205000 // 512 + 64
    assert n >= pairs * 32 * (128 + 2) * 4
    assert n < 2 * pairs * 32 * (128 + 2) * 4 + 64 * 16 + 4096
    loose = f(64, 64, 1, 16384, -1, 32, 8, 128, 16, 1)
    assert loose >= n
    # unsupported geometry -> 0
    assert f(1, 1, 1, 16, 16, 32, 8, 96, 16, 1) == 0
    assert f(1, 1, 1, 16, 16, 32, 8, 128, 8, 1) == 0
    assert f(1, 1, 1, 16, 16, 30, 8, 128, 16, 1) == 0
    assert f(1, 1, 1, 16, 16, 32, 8, 128, 16, 7) == 0
    assert f(1, 1, 1, 16, 16, 34, 2, 128, 16, 1) == 0  # group of 17 heads


def _attn(lib, **kw):
    a = dict(q=1 << 12, kc=1 << 12, vc=1 << 12, bt=1 << 12, mb=4, cu=1 << 12, ctx=1 << 12,
             slot=None, kn=None, vn=None, out=1 << 12, B=1, T=1, H=4, Hkv=2, D=64, bs=16,
             NB=8, mq=1, mc=16, scale=0.125, dt=0, ws=1 << 12, wsb=1 << 20, st=None, stream=None)
    a.update(kw)
    return lib.pa_attention(a["q"], a["kc"], a["vc"], a["bt"], a["mb"], a["cu"], a["ctx"],
                            a["slot"], a["kn"], a["vn"], a["out"], a["B"], a["T"], a["H"],
                            a["Hkv"], a["D"], a["bs"], a["NB"], a["mq"], a["mc"], a["scale"],
                            a["dt"], a["ws"], a["wsb"], a["st"], a["stream"])


def test_attention_refusals_before_cuda(lib):
    # every case fails validation, so no CUDA call is made on this GPU-less host
    assert _attn(lib, D=96) == 2
    assert _attn(lib, bs=8) == 2
    assert _attn(lib, H=6, Hkv=4) == 2
    assert _attn(lib, dt=5) == 2
    assert _attn(lib, q=None) == 1
    assert _attn(lib, out=None) == 1
    assert _attn(lib, B=-1) == 1
    assert _attn(lib, T=-1) == 1
    assert _attn(lib, NB=0) == 1
    assert _attn(lib, mb=0) == 1
    assert _attn(lib, q=(1 << 12) + 4) == 1  # misaligned
    assert _attn(lib, slot=1 << 12) == 1  # write args must come together
    assert _attn(lib, scale=float("nan")) == 1
    assert _attn(lib, scale=0.0) == 1
    assert _attn(lib, scale=-0.125) == 1
    assert _attn(lib, ws=None) == 3
    assert _attn(lib, ws=(1 << 12) + 16) == 3  # workspace not 256-byte aligned
    assert _attn(lib, wsb=64) == 3  # too small for even one split
    assert _attn(lib, T=1, B=0) == 1
    assert _attn(lib, NB=1 << 27, bs=32) == 2  # token coordinate would overflow int32


def test_write_refusals_before_cuda(lib):
    f = lib.pa_write_kv
    assert f(None, None, None, None, None, 0, 8, 16, 2, 64, 0, None, None) == 0  # nothing to do
    assert f(None, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 3, 8, 16, 2, 64, 0, None, None) == 1
    assert f(1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 3, 8, 16, 2, 96, 0, None, None) == 2
    assert f(1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 3, 0, 16, 2, 64, 0, None, None) == 1
    assert f(1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, -1, 8, 16, 2, 64, 0, None, None) == 1


def test_no_launches_counted_on_refusals(lib):
    before = lib.pa_kernel_launches()
    _attn(lib, D=96)
    assert lib.pa_kernel_launches() == before


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        pa.load()


def test_workspace_bytes_ex_modes(lib):
    f = lib.pa_attention_workspace_bytes_ex
    args = (128, 4216, 512, 16384, 120 * 3000 + 8 * 2560, 40, 8, 128, 16, 1)
    batch = f(*args, 0)
    row = f(*args, 1)
    assert batch == lib.pa_attention_workspace_bytes(*args)
    # row mode: every row holds up to ceil(max_ctx / 512) splits
    pairs = 4216 * (16384 // 512)
    assert row >= pairs * 40 * (128 + 2) * 4
    assert row > batch
    # fp32 steps split every row in both modes
    f32 = args[:-1] + (0,)
    assert f(*f32, 0) == f(*f32, 1)
    assert f(*args, 2) == 0 and f(*args, -1) == 0  # unknown mode
    # the reuse-plan bit sizes nothing; other bits are unknown
    assert f(*args, 0x100) == batch and f(*args, 0x101) == row
    assert f(*args, 0x200) == 0 and f(*args, 0x102) == 0 and f(*args, 0x300) == 0


def test_attention_ex_refuses_unknown_mode(lib):
    a = [1 << 12, 1 << 12, 1 << 12, 1 << 12, 4, 1 << 12, 1 << 12, None, None, None, 1 << 12,
         1, 1, 4, 2, 64, 16, 8, 1, 16, 0.125, 0, 1 << 12, 1 << 20, None, None]
    before = lib.pa_kernel_launches()
    assert lib.pa_attention_ex(*a, 1.0, 1.0, 2, None, 0) == 1
    assert lib.pa_attention_ex(*a, 1.0, 1.0, -1, None, 0) == 1
    for bad in (0x200, 0x102, 0x301):  # only an invariance mode and the reuse bit are known
        assert lib.pa_attention_ex(*a, 1.0, 1.0, bad, None, 0) == 1
    assert lib.pa_attention_ex(*(a[:15] + [96] + a[16:]), 1.0, 1.0, 1, None, 0) == 2
    assert lib.pa_kernel_launches() == before


def test_e4m3_refusals_before_cuda(lib):
    a = [1 << 12, 1 << 12, 1 << 12, 1 << 12, 4, 1 << 12, 1 << 12, None, None, None, 1 << 12,
         1, 1, 4, 2, 64, 16, 8, 1, 16, 0.125, 2, 1 << 12, 1 << 20, None, None]
    before = lib.pa_kernel_launches()
    # the base entry points have no scales
    assert lib.pa_attention(*a) == 2
    assert lib.pa_write_kv(1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 3, 8, 16, 2, 64, 2,
                           None, None) == 2
    # scales must be finite and positive
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert lib.pa_attention_ex(*a, ks, vs, 0, None, 0) == 1
        assert lib.pa_write_kv_scaled(1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 3, 8, 16, 2,
                                      64, 2, ks, vs, None, None) == 1
    # other types ignore the scales
    assert lib.pa_write_kv_scaled(None, None, None, None, None, 0, 8, 16, 2, 64, 1, 0.0, 0.0,
                                  None, None) == 0
    assert lib.pa_kernel_launches() == before
    # workspace: e4m3 steps split every row, in either mode
    f = lib.pa_attention_workspace_bytes_ex
    args = (16, 600, 512, 4096, 10000, 32, 8, 128, 16, 2)
    assert f(*args, 0) == f(*args, 1) == f(*(args[:-1] + (0,)), 0)


def test_kv_parallel_refusals_before_cuda(lib):
    before = lib.pa_kernel_launches()
    pb = lib.pa_partials_bytes(64, 4096, 32, 128)
    assert pb >= 64 * 8 * 32 * (128 + 2) * 4 and pb % 256 == 0
    assert lib.pa_partials_bytes(64, 4096, 32, 96) == 0
    ws = lib.pa_partials_workspace_bytes(8, 64, 4096)
    assert ws > 64 * 8 * 16
    base = [1 << 12, 1 << 12, 1 << 12, 1 << 12, 4, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 1, 1, 4,
            2, 64, 16, 8, 1, 16, 0.125, 0, 1.0, 1.0, 1 << 12, 1 << 20, 1 << 12, 1 << 20, None,
            None]
    f = lib.pa_attention_partials
    assert f(*(base[:7] + [None] + base[8:])) == 1          # key_lo missing
    assert f(*(base[:13] + [96] + base[14:])) == 2          # D unsupported
    assert f(*(base[:22] + [(1 << 12) + 16] + base[23:])) == 3  # partials misaligned
    assert f(*(base[:23] + [64] + base[24:])) == 3          # partials too small
    assert f(*(base[:25] + [16] + base[26:])) == 3          # workspace too small
    m = lib.pa_merge_partials
    mb = [1 << 12, 1 << 20, 2, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 1, 1, 4, 64, 1, 16, 0, 1.0,
          1 << 12, 1 << 20, None, None]
    assert m(*(mb[:2] + [0] + mb[3:])) == 1                  # no owners
    assert m(*(mb[:3] + [None] + mb[4:])) == 1               # no bounds
    assert m(*(mb[:1] + [1 << 20 | 8] + mb[2:])) == 3        # owner stride not 256-aligned
    assert lib.pa_kernel_launches() == before


def test_decode_gemm_refusals_before_cuda(lib):
    before = lib.pa_kernel_launches()
    f = lib.pa_decode_gemm
    assert f(1 << 12, 1 << 12, 1 << 12, 48, 1024, 5120, None, 0, None, None) == 2   # T_pad
    assert f(1 << 12, 1 << 12, 1 << 12, 64, 1000, 5120, None, 0, None, None) == 2   # N % 128
    assert f(1 << 12, 1 << 12, 1 << 12, 64, 1024, 5000, None, 0, None, None) == 2   # K % 64
    assert f(None, 1 << 12, 1 << 12, 64, 1024, 5120, None, 0, None, None) == 1
    assert f(1 << 12, 1 << 12, (1 << 12) + 2, 64, 1024, 5120, None, 0, None, None) == 1
    assert f(1 << 12, 1 << 12, 1 << 12, 64, 1024, 5120, None, 0, None, None) == 3   # needs split-K scratch
    assert lib.pa_kernel_launches() == before
    # the plan is a function of the shape only
    assert lib.pa_decode_gemm_splits(1024, 5120) == 20
    assert lib.pa_decode_gemm_splits(248320, 5120) == 1
    assert lib.pa_decode_gemm_workspace_bytes(64, 248320, 5120) == 0
    assert lib.pa_decode_gemm_workspace_bytes(64, 1024, 5120) >= 20 * 64 * 1024 * 4


def test_static_scratch_refusals_before_cuda(lib):
    """Negative sizes are refused as pa_attention refuses them (invalid
    argument), a step beyond the built-in array as a workspace error, and
    unsupported geometry as unsupported -- all before any CUDA call."""
    f = lib.pa_attention_static_scratch

    def call(B=4, T=4, H=8, Hkv=2, D=128, bs=16, NB=64, mq=1, mc=40, tot=69):
        return f(None, None, None, None, 3, None, None, None, None, None, None, B, T, H, Hkv,
                 D, bs, NB, mq, mc, tot, 0.088, 1, None, None)
    assert call(B=-1) == 1
    assert call(T=-1) == 1
    assert call(mq=-1) == 1
    assert call(mc=-1) == 1
    assert call(NB=0) == 1
    assert call(D=96) == 2
    assert call(B=256, T=256, H=64, Hkv=8, mc=40960, tot=10 ** 7) == 3
