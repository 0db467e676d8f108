"""The C-ABI library builds, loads, exports every declared symbol, and rejects
bad arguments on the host before touching a GPU (no compute calls here)."""

import ctypes
import os
import re

import pytest

from _util import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    with open(os.path.join(ROOT, "include", "fattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from exact_attention_06_gb300 import fattn
    return fattn.lib()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("fa_fwd", "fa_fwd_ex", "fa_fwd_fp8", "fa_quantize_e4m3", "fa_decode_splitkv",
              "fa_decode_workspace_bytes", "fa_combine",
              "fa_get_status", "fa_status_string", "fa_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from exact_attention_06_gb300 import fattn
    names = _declared_functions()
    assert sorted(fattn.EXPORTED) == names
    for n in names:
        assert hasattr(lib, n), f"libfattn.so does not export {n}"


def test_status_strings(lib):
    from exact_attention_06_gb300 import fattn
    assert fattn.status_string(0) == "FA_OK"
    assert fattn.status_string(fattn.FA_ERR_TIMEOUT) == "FA_ERR_TIMEOUT"
    assert fattn.status_string(99) == "FA_ERR_UNKNOWN"


def _fwd(lib, ptrs=(16, 16, 16, 16, 16), B=1, H=1, N=8, d=64, scale=0.125, causal=0):
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(ptrs[0]), vp(ptrs[1]), vp(ptrs[2]), vp(ptrs[3]), vp(ptrs[4]), B, H, N, d,
                      ctypes.c_float(scale), causal, vp(0))


def test_forward_argument_checks_need_no_gpu(lib):
    from exact_attention_06_gb300 import fattn
    assert _fwd(lib, ptrs=(0, 16, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG
    assert _fwd(lib, N=0) == fattn.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=-1) == fattn.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == fattn.FA_ERR_UNSUPPORTED
    assert _fwd(lib, scale=float("nan")) == fattn.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=0.0) == fattn.FA_ERR_INVALID_ARG
    assert _fwd(lib, causal=2) == fattn.FA_ERR_INVALID_ARG
    assert _fwd(lib, ptrs=(16, 24, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # misaligned k
    assert _fwd(lib, ptrs=(16, 16, 16, 16, 18)) == fattn.FA_ERR_INVALID_ARG  # misaligned lse
    assert _fwd(lib, N=65535 * 128 + 1) == fattn.FA_ERR_UNSUPPORTED
    assert "aligned" in fattn.fa_last_error() or "N=" in fattn.fa_last_error()


def test_forward_workspace_query_without_a_split(lib):
    # invalid sizes and causal launches plan no split (with or without a device)
    lib.fa_fwd_workspace_bytes.restype = ctypes.c_size_t
    assert lib.fa_fwd_workspace_bytes(0, 1, 2048, 64, 0) == 0
    assert lib.fa_fwd_workspace_bytes(1, 1, 2048, 96, 0) == 0
    assert lib.fa_fwd_workspace_bytes(1, 1, 2048, 64, 2) == 0
    assert lib.fa_fwd_workspace_bytes(4, 16, 2048, 64, 1) == 0


def test_backward_workspace_and_options_need_no_gpu(lib):
    """fa_bwd_workspace_bytes is D's size (B*H*N fp32, 256-byte rounded); fa_bwd_ex with options
    and fa_bwd reject a too small workspace and an unsupported d before any device call."""
    from exact_attention_06_gb300 import fattn
    vp, f = ctypes.c_void_p, ctypes.c_float
    assert fattn.fa_bwd_workspace_bytes(2, 16, 8192) == 2 * 16 * 8192 * 4
    assert fattn.fa_bwd_workspace_bytes(1, 1, 3) == 256
    assert fattn.fa_bwd_workspace_bytes(0, 1, 3) == 0
    need = fattn.fa_bwd_workspace_bytes(1, 1, 256)
    ptrs = [vp(256)] * 9
    opts = fattn.FaBwdOpts(1000)

    def bwd_ex(ws_bytes, d=128, o=ctypes.byref(opts)):
        return lib.fa_bwd_ex(*ptrs, 1, 1, 256, d, f(0.1), 1, 0, vp(256), ws_bytes, vp(0), o)

    assert bwd_ex(need - 1) == fattn.FA_ERR_WORKSPACE
    assert bwd_ex(need - 1, o=None) == fattn.FA_ERR_WORKSPACE
    assert bwd_ex(need, d=96) == fattn.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd(*ptrs, 1, 1, 256, 128, f(0.1), 1, 0, vp(256), need - 1, vp(0)) == fattn.FA_ERR_WORKSPACE


def test_decode_workspace_sizes(lib):
    from exact_attention_06_gb300 import fattn
    # explicit splits need no device: R*S*d floats + R*S + R*S floats, each rounded up to 256 bytes
    assert fattn.fa_decode_workspace_bytes(64, 32, 32768, 128, 128, 4) == 2048 * 4 * 128 * 4 + 2 * 2048 * 4 * 4
    assert fattn.fa_decode_workspace_bytes(1, 1, 1, 64, 128, 1) == 256 * 3
    assert fattn.fa_decode_workspace_bytes(1, 1, 1000, 64, 128, 9) == 0  # more splits than 128-key chunks
    assert fattn.fa_decode_workspace_bytes(1, 1, 1000, 64, 64, 1) == 0   # chunk must be 128
    assert fattn.fa_decode_workspace_bytes(1, 1, 1000, 80, 128, 1) == 0
    assert fattn.fa_decode_workspace_bytes(1, 1, 0, 64, 128, 1) == 0


def test_decode_and_combine_argument_checks_need_no_gpu(lib):
    from exact_attention_06_gb300 import fattn
    vp, f = ctypes.c_void_p, ctypes.c_float
    st = lib.fa_decode_splitkv(vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, 256, 128, f(0.1), 128, 1, vp(256),
                               ctypes.c_size_t(16), vp(0))
    assert st == fattn.FA_ERR_WORKSPACE
    st = lib.fa_decode_splitkv(vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, 256, 128, f(0.1), 128, 3, vp(256),
                               ctypes.c_size_t(1 << 20), vp(0))
    assert st == fattn.FA_ERR_INVALID_ARG  # 3 splits > 2 chunks
    st = lib.fa_decode_splitkv(vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, 256, 128, f(0.1), 128, 1, vp(264),
                               ctypes.c_size_t(1 << 20), vp(0))
    assert st == fattn.FA_ERR_INVALID_ARG  # workspace not 256-byte aligned
    st = lib.fa_combine(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 0, 128, vp(0))
    assert st == fattn.FA_ERR_INVALID_ARG
    st = lib.fa_combine(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 2, 32, vp(0))
    assert st == fattn.FA_ERR_UNSUPPORTED


def test_decode_and_combine_options_are_checked_before_any_launch(lib):
    """The _ex entry points reject a bad o_fp32 flag (and everything the plain calls reject)
    before touching a GPU; a NULL options pointer means the defaults."""
    from exact_attention_06_gb300 import fattn
    vp, f, sz = ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
    bad = fattn.FaDecodeOpts(2, 0)
    st = lib.fa_decode_splitkv_ex(vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, 256, 128, f(0.1), 128, 1, vp(256),
                                  sz(1 << 20), vp(0), ctypes.byref(bad))
    assert st == fattn.FA_ERR_INVALID_ARG and "o_fp32" in fattn.fa_last_error()
    st = lib.fa_decode_splitkv_ex(vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, 256, 128, f(0.1), 128, 1, vp(256),
                                  sz(16), vp(0), None)
    assert st == fattn.FA_ERR_WORKSPACE
    st = lib.fa_decode_paged_ex(vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), 1, 1, 128, 64, 4, 4, 256,
                                f(0.1), 0, vp(256), sz(1 << 20), vp(0), ctypes.byref(bad))
    assert st == fattn.FA_ERR_INVALID_ARG and "o_fp32" in fattn.fa_last_error()
    assert lib.fa_combine_ex(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 2, 128, 2, vp(0)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_combine_ex(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 0, 128, 1, vp(0)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_combine_ex(vp(16), vp(16), vp(16), vp(8), vp(16), 4, 2, 128, 1, vp(0)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_combine_ex(vp(16), vp(16), vp(16), vp(16), vp(16), 4, 2, 96, 0, vp(0)) == fattn.FA_ERR_UNSUPPORTED


def test_fp8_argument_checks_need_no_gpu(lib):
    from exact_attention_06_gb300 import fattn
    vp, f = ctypes.c_void_p, ctypes.c_float

    def fwd8(ptrs=(16,) * 8, N=256, d=128, scale=0.1, causal=0):
        return lib.fa_fwd_fp8(*(vp(p) for p in ptrs), 1, 2, N, d, f(scale), causal, vp(0), None)

    assert fwd8(d=64) == fattn.FA_ERR_UNSUPPORTED  # FP8 forward is d = 128 only
    assert fwd8(ptrs=(16, 16, 16, 0, 16, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # null scale array
    assert fwd8(ptrs=(16, 16, 8, 16, 16, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # misaligned v8
    assert fwd8(ptrs=(16, 16, 16, 16, 18, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # misaligned sk
    assert fwd8(N=0) == fattn.FA_ERR_INVALID_ARG
    assert fwd8(scale=-1.0) == fattn.FA_ERR_INVALID_ARG
    assert fwd8(causal=3) == fattn.FA_ERR_INVALID_ARG
    q = lib.fa_quantize_e4m3
    assert q(vp(16), vp(16), vp(16), 1, 1, 128, 96, vp(0)) == fattn.FA_ERR_UNSUPPORTED
    assert q(vp(16), vp(24), vp(16), 1, 1, 128, 128, vp(0)) == fattn.FA_ERR_INVALID_ARG  # codes misaligned
    assert q(vp(16), vp(16), vp(0), 1, 1, 128, 128, vp(0)) == fattn.FA_ERR_INVALID_ARG
    assert q(vp(16), vp(16), vp(16), 1, 0, 128, 128, vp(0)) == fattn.FA_ERR_INVALID_ARG


def test_paged_decode_argument_checks_need_no_gpu(lib):
    from exact_attention_06_gb300 import fattn
    vp, f, sz = ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t

    def paged(ptrs=(16,) * 7, B=2, H=4, d=128, page_size=128, max_pages=8, num_pages=16, max_seq_len=1000,
              scale=0.1, splits=1, ws=256, ws_bytes=1 << 20):
        return lib.fa_decode_paged(*(vp(p) for p in ptrs), B, H, d, page_size, max_pages, num_pages, max_seq_len,
                                   f(scale), splits, vp(ws), sz(ws_bytes), vp(0))

    assert paged(page_size=96) == fattn.FA_ERR_UNSUPPORTED      # not a multiple of 64
    assert paged(page_size=0) == fattn.FA_ERR_UNSUPPORTED
    assert paged(d=80) == fattn.FA_ERR_UNSUPPORTED
    assert paged(max_seq_len=8 * 128 + 1) == fattn.FA_ERR_INVALID_ARG  # more than max_pages * page_size
    assert paged(max_seq_len=0) == fattn.FA_ERR_INVALID_ARG
    assert paged(num_pages=0) == fattn.FA_ERR_INVALID_ARG
    assert paged(ptrs=(16, 16, 16, 0, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # null block table
    assert paged(ptrs=(16, 16, 16, 18, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # misaligned block table
    assert paged(ptrs=(16, 24, 16, 16, 16, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # misaligned k pool
    assert paged(splits=-1) == fattn.FA_ERR_INVALID_ARG
    assert paged(splits=9) == fattn.FA_ERR_INVALID_ARG            # more splits than 128-key chunks
    assert paged(ws_bytes=16) == fattn.FA_ERR_WORKSPACE
    # explicit splits: the workspace size needs no device and matches the contiguous decode's
    assert fattn.fa_decode_paged_workspace_bytes(2, 4, 1000, 128, 128, 8, 2) == \
        fattn.fa_decode_workspace_bytes(2, 4, 1000, 128, 128, 2)
    assert fattn.fa_decode_paged_workspace_bytes(2, 4, 1000, 128, 100, 8, 2) == 0
    # a split may cover at most 1023 pages: one split over 70000 keys of 64-key pages is refused
    assert fattn.fa_decode_paged_workspace_bytes(1, 1, 70000, 64, 64, 1100, 1) == 0
    assert paged(page_size=64, max_pages=1100, max_seq_len=70000, splits=1, ws_bytes=1 << 30) == \
        fattn.FA_ERR_UNSUPPORTED


def test_partial_forward_argument_checks_need_no_gpu(lib):
    from exact_attention_06_gb300 import fattn
    vp, f = ctypes.c_void_p, ctypes.c_float

    def part(ptrs=(16,) * 6, N=256, Nk=128, koff=0, d=128, shard=0, S=2, causal=1):
        return lib.fa_fwd_partial(*(vp(p) for p in ptrs), 1, 2, N, Nk, koff, d, f(0.1), causal, shard, S, vp(0))

    assert part(shard=2) == fattn.FA_ERR_INVALID_ARG
    assert part(shard=-1) == fattn.FA_ERR_INVALID_ARG
    assert part(S=0) == fattn.FA_ERR_INVALID_ARG
    assert part(koff=-5) == fattn.FA_ERR_INVALID_ARG
    assert part(Nk=0) == fattn.FA_ERR_INVALID_ARG
    assert part(d=96) == fattn.FA_ERR_UNSUPPORTED
    assert part(ptrs=(16, 16, 16, 8, 16, 16)) == fattn.FA_ERR_INVALID_ARG  # u_part misaligned
    assert part(ptrs=(16, 16, 16, 16, 0, 16)) == fattn.FA_ERR_INVALID_ARG


def test_partial_forward_key_range_checks_need_no_gpu(lib):
    from exact_attention_06_gb300 import fattn
    vp, f = ctypes.c_void_p, ctypes.c_float

    def part(Nk=100, key_offset=200, kv_rows=300):
        return lib.fa_fwd_partial_ex(*(vp(16) for _ in range(6)), 1, 1, 256, Nk, key_offset, kv_rows, 64, f(0.1), 1,
                                     0, 2, vp(0))

    assert part(kv_rows=299) == fattn.FA_ERR_INVALID_ARG  # the shard ends past the tensor
    assert part(kv_rows=-1) == fattn.FA_ERR_INVALID_ARG
    assert part(key_offset=-1) == fattn.FA_ERR_INVALID_ARG
    assert "kv_rows" in fattn.fa_last_error() or "key_offset" in fattn.fa_last_error()


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    # no fallback: a missing libfattn.so is an error, not a silent CPU path
    from exact_attention_06_gb300 import fattn
    monkeypatch.setattr(fattn, "_lib", None)
    monkeypatch.setattr(fattn, "LIB_PATH", str(tmp_path / "libfattn.so"))
    with pytest.raises(fattn.FattnError) as ei:
        fattn.lib()
    assert "missing" in str(ei.value)


def test_binding_rejects_tensors_the_library_cannot_read(lib):
    """The binding passes raw device pointers, so it refuses host tensors, strided views, wrong
    dtypes and mismatched shapes with FA_ERR_INVALID_ARG before anything reaches the library."""
    import torch
    from exact_attention_06_gb300 import fattn
    B, H, N, d = 1, 2, 16, 64
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    lse = torch.zeros(B, H, N, dtype=torch.float32)

    def rejected(fn, *args, what, **kw):
        with pytest.raises(fattn.FattnError) as err:
            fn(*args, **kw)
        assert err.value.status == fattn.FA_ERR_INVALID_ARG
        assert what in str(err.value), str(err.value)

    # (the checks run in argument order and each tensor is checked for dtype, shape, layout and
    # device in turn; the tensors here are on the host, so the faulty one goes first)
    rejected(fattn.fa_fwd, q, q, q, q, lse, 0.1, what="CUDA tensor")
    rejected(fattn.fa_fwd, q.transpose(2, 3).contiguous().transpose(2, 3), q, q, q, lse, 0.1, what="contiguous")
    rejected(fattn.fa_fwd, q.float(), q, q, q, lse, 0.1, what="dtype")
    k = torch.zeros(B, H, N // 2, d, dtype=torch.bfloat16)
    rejected(fattn.fa_fwd_partial, q.float(), k, k, torch.zeros(B * H * N, 2, d), torch.zeros(B * H * N, 2),
             torch.zeros(B * H * N, 2), 0.1, 0, 0, what="dtype")
    rejected(fattn.fa_decode_splitkv, q[:, :, 0], q, q, q[:, :, 0].contiguous(), lse[:, :, 0].contiguous(), 0.1,
             torch.zeros(256, dtype=torch.uint8), what="q must be contiguous")
    u = torch.zeros(4, 2, d)
    m = torch.zeros(4, 2)
    rejected(fattn.fa_combine, u.double(), m, m, torch.zeros(4, d), torch.zeros(4), what="u_part")
    rejected(fattn.fa_decode_splitkv, q[:, :1, 0].contiguous(), q, q, q[:, :, 0].contiguous(),
             lse[:, :, 0].contiguous(), 0.1, torch.zeros(256, dtype=torch.uint8), what="shape")
    rejected(fattn.fa_decode_paged, q[:, :, 0].contiguous().float(), q, q, torch.zeros(1, 4, dtype=torch.int32),
             torch.zeros(1, dtype=torch.int32), q[:, :, 0].contiguous(), lse[:, :, 0].contiguous(), 0.1, 64,
             workspace=torch.zeros(256, dtype=torch.uint8), what="dtype")
