"""Thin ctypes binding of the libfattn C ABI (include/fattn.h).

Argument marshalling only: every function takes torch CUDA tensors (or sizes),
passes their device pointers and the current CUDA stream to the function of
the same name in ``libfattn.so`` and raises ``FattnError`` on a non-OK status.
All computation happens in the library's kernels; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfattn.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ARCH = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_ERR_WORKSPACE = 6

# Every symbol include/fattn.h declares.
EXPORTED = ("fa_fwd", "fa_fwd_ex", "fa_fwd_workspace_bytes", "fa_fwd_partial", "fa_fwd_partial_ex",
            "fa_quantize_e4m3", "fa_fwd_fp8",
            "fa_bwd_workspace_bytes", "fa_bwd", "fa_bwd_ex", "fa_decode_workspace_bytes", "fa_decode_splitkv",
            "fa_decode_splitkv_ex", "fa_decode_splitkv_noalloc", "fa_decode_paged_workspace_bytes",
            "fa_decode_paged", "fa_decode_paged_ex", "fa_combine", "fa_combine_ex", "fa_get_status",
            "fa_status_string", "fa_last_error")
FA_NOALLOC_SCRATCH_BYTES = 8 << 20


class FattnError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        self.status = status
        super().__init__(f"{func}: {status_string(status)}: {detail}")


class FaFwdOpts(ctypes.Structure):
    _fields_ = [("o_fp32", ctypes.c_int), ("wait_budget_cycles", ctypes.c_ulonglong),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class FaDecodeOpts(ctypes.Structure):
    _fields_ = [("o_fp32", ctypes.c_int), ("wait_budget_cycles", ctypes.c_ulonglong)]


class FaBwdOpts(ctypes.Structure):
    _fields_ = [("wait_budget_cycles", ctypes.c_ulonglong)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FattnError(FA_ERR_CUDA, "load", f"{LIB_PATH} is missing; build it with exact_attention_06_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, ctypes.POINTER(FaFwdOpts)]
        L.fa_fwd_workspace_bytes.argtypes = [i, i, i, i, i]
        L.fa_fwd_workspace_bytes.restype = sz
        L.fa_fwd_partial.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, i, vp]
        L.fa_fwd_partial_ex.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp]
        L.fa_quantize_e4m3.argtypes = [vp, vp, vp, i, i, i, i, vp]
        L.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, ctypes.POINTER(FaFwdOpts)]
        L.fa_bwd_workspace_bytes.argtypes = [i, i, i]
        L.fa_bwd_workspace_bytes.restype = sz
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
        L.fa_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp,
                                ctypes.POINTER(FaBwdOpts)]
        L.fa_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
        L.fa_decode_workspace_bytes.restype = sz
        L.fa_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
        L.fa_decode_splitkv_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp,
                                           ctypes.POINTER(FaDecodeOpts)]
        L.fa_decode_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        L.fa_decode_paged_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        L.fa_decode_paged_workspace_bytes.restype = sz
        L.fa_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
        L.fa_decode_paged_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp,
                                         ctypes.POINTER(FaDecodeOpts)]
        L.fa_combine.argtypes = [vp, vp, vp, vp, vp, i, i, i, vp]
        L.fa_combine_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
        L.fa_get_status.argtypes = [vp]
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_last_error.argtypes = []
        L.fa_last_error.restype = ctypes.c_char_p
        for name in ("fa_fwd", "fa_fwd_ex", "fa_fwd_partial", "fa_fwd_partial_ex", "fa_quantize_e4m3", "fa_fwd_fp8",
                     "fa_bwd", "fa_bwd_ex",
                     "fa_decode_splitkv", "fa_decode_splitkv_ex", "fa_decode_splitkv_noalloc", "fa_decode_paged",
                     "fa_decode_paged_ex", "fa_combine", "fa_combine_ex", "fa_get_status"):
            getattr(L, name).restype = i
        _lib = L
    return _lib


_STATUS_NAMES = {FA_OK: "FA_OK", FA_ERR_INVALID_ARG: "FA_ERR_INVALID_ARG", FA_ERR_UNSUPPORTED: "FA_ERR_UNSUPPORTED",
                 FA_ERR_ARCH: "FA_ERR_ARCH", FA_ERR_CUDA: "FA_ERR_CUDA", FA_ERR_TIMEOUT: "FA_ERR_TIMEOUT",
                 FA_ERR_WORKSPACE: "FA_ERR_WORKSPACE"}


def status_string(status: int) -> str:
    """The library's name for a status; the enum's name when the library is not loaded
    (so that the error raised for a missing library can be built)."""
    if _lib is None:
        return _STATUS_NAMES.get(int(status), "FA_ERR_UNKNOWN")
    return _lib.fa_status_string(int(status)).decode()


def fa_status_string(status: int) -> str:
    return status_string(status)


def fa_last_error() -> str:
    return lib().fa_last_error().decode()


def _check(status: int, func: str):
    if status != FA_OK:
        raise FattnError(status, func, fa_last_error())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


_BF16 = (torch.bfloat16,)
_F32 = (torch.float32,)
_OUT = (torch.bfloat16, torch.float32)
_U8 = (torch.uint8,)
_I32 = (torch.int32,)


def _need(func: str, name: str, t, dtypes, shape=None):
    """The library reads and writes plain contiguous device buffers: refuse anything else here,
    before a pointer is passed (a strided view or a host tensor would be read as garbage)."""
    if not isinstance(t, torch.Tensor):
        raise FattnError(FA_ERR_INVALID_ARG, func, f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise FattnError(FA_ERR_INVALID_ARG, func, f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise FattnError(FA_ERR_INVALID_ARG, func, f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise FattnError(FA_ERR_INVALID_ARG, func, f"{name} must be contiguous")
    if not t.is_cuda:
        raise FattnError(FA_ERR_INVALID_ARG, func, f"{name} must be a CUDA tensor")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def fa_fwd_workspace_bytes(B: int, H: int, N: int, d: int, causal: bool = False) -> int:
    """Scratch bytes of the key split of fa_fwd_ex's last round on the current device (0: no key split)."""
    return int(lib().fa_fwd_workspace_bytes(B, H, N, d, int(bool(causal))))


def fa_fwd_ex(q, k, v, o, lse, scale: float, causal: bool = False, stream=None, o_fp32: bool | None = None,
              wait_budget_cycles: int = 0, workspace=None):
    """Fused forward: q, k, v, o [B, H, N, d]; lse [B, H, N] fp32.

    ``o`` may be bf16 (default) or fp32 (``o_fp32``, inferred from o's dtype).  ``workspace``:
    an optional uint8 CUDA tensor of at least fa_fwd_workspace_bytes() bytes for the key split.
    """
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need("fa_fwd_ex", name, t, _BF16, (B, H, N, d))
    _need("fa_fwd_ex", "o", o, _OUT, (B, H, N, d))
    _need("fa_fwd_ex", "lse", lse, _F32, (B, H, N))
    if workspace is not None:
        _need("fa_fwd_ex", "workspace", workspace, _U8)
    if o_fp32 is None:
        o_fp32 = o.dtype == torch.float32
    elif bool(o_fp32) != (o.dtype == torch.float32):
        raise FattnError(FA_ERR_INVALID_ARG, "fa_fwd_ex", f"o_fp32={o_fp32} but o has dtype {o.dtype}")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    opts = FaFwdOpts(int(bool(o_fp32)), int(wait_budget_cycles), _ptr(workspace) if workspace is not None else None,
                     ws_bytes)
    st = lib().fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(bool(causal)),
                         _stream(stream), ctypes.byref(opts))
    _check(st, "fa_fwd_ex")


def fa_fwd(q, k, v, o, lse, scale: float, causal: bool = False, stream=None):
    """Fused forward with bf16 O (see fa_fwd_ex)."""
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _need("fa_fwd", name, t, _BF16, (B, H, N, d))
    _need("fa_fwd", "lse", lse, _F32, (B, H, N))
    st = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(bool(causal)),
                      _stream(stream))
    _check(st, "fa_fwd")


def fa_fwd_partial(q, k, v, u_part, m_part, l_part, scale: float, key_offset: int, shard: int,
                   causal: bool = False, stream=None, nk: int | None = None):
    """Forward over one key shard: q [B, H, N, d]; writes slot ``shard`` of u_part [B*H*N, S, d],
    m_part / l_part [B*H*N, S] fp32.  k, v are the shard's own [B, H, Nk, d] buffers (global key
    indices from key_offset), or, with ``nk``, the whole [B, H, L, d] key tensors of which the
    shard is rows key_offset .. key_offset + nk - 1 (fa_fwd_partial_ex, no copy)."""
    B, H, N, d = q.shape
    _need("fa_fwd_partial", "q", q, _BF16, (B, H, N, d))
    _need("fa_fwd_partial", "k", k, _BF16, (B, H, k.shape[2], d))
    _need("fa_fwd_partial", "v", v, _BF16, tuple(k.shape))
    S = u_part.shape[1]
    _need("fa_fwd_partial", "u_part", u_part, _F32, (B * H * N, S, d))
    _need("fa_fwd_partial", "m_part", m_part, _F32, (B * H * N, S))
    _need("fa_fwd_partial", "l_part", l_part, _F32, (B * H * N, S))
    kv_rows = 0 if nk is None else k.shape[2]
    Nk = k.shape[2] if nk is None else int(nk)
    st = lib().fa_fwd_partial_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(u_part), _ptr(m_part), _ptr(l_part), B, H, N, Nk,
                                 int(key_offset), kv_rows, d, float(scale), int(bool(causal)), int(shard), S,
                                 _stream(stream))
    _check(st, "fa_fwd_partial_ex")


def fa_quantize_e4m3(x, codes, scales, stream=None):
    """E4M3 block quantization: x [B, H, N, d] bf16 -> codes [B, H, N, d] uint8, scales [B, H, ceil(N/128)] fp32."""
    B, H, N, d = x.shape
    _need("fa_quantize_e4m3", "x", x, _BF16)
    _need("fa_quantize_e4m3", "codes", codes, _U8, (B, H, N, d))
    _need("fa_quantize_e4m3", "scales", scales, _F32, (B, H, (N + 127) // 128))
    st = lib().fa_quantize_e4m3(_ptr(x), _ptr(codes), _ptr(scales), B, H, N, d, _stream(stream))
    _check(st, "fa_quantize_e4m3")


def fa_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, scale: float, causal: bool = False, stream=None,
               wait_budget_cycles: int = 0):
    """FP8 forward: q8, k8, v8 [B, H, N, 128] uint8 E4M3 codes with block scales sq, sk, sv
    [B, H, ceil(N/128)] fp32; o [B, H, N, 128] bf16 or fp32 (from its dtype); lse [B, H, N] fp32."""
    B, H, N, d = q8.shape
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        _need("fa_fwd_fp8", name, t, _U8, (B, H, N, d))
    for name, t in (("sq", sq), ("sk", sk), ("sv", sv)):
        _need("fa_fwd_fp8", name, t, _F32, (B, H, (N + 127) // 128))
    _need("fa_fwd_fp8", "o", o, _OUT, (B, H, N, d))
    _need("fa_fwd_fp8", "lse", lse, _F32, (B, H, N))
    opts = FaFwdOpts(int(o.dtype == torch.float32), int(wait_budget_cycles))
    st = lib().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o), _ptr(lse), B, H, N, d,
                          float(scale), int(bool(causal)), _stream(stream), ctypes.byref(opts))
    _check(st, "fa_fwd_fp8")


def fa_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scale: float, causal: bool = False, workspace=None, stream=None,
           wait_budget_cycles: int = 0):
    """Backward: gradients dq, dk, dv (bf16 or fp32, from dq's dtype) of the forward that produced o, lse.
    A non-zero wait_budget_cycles calls fa_bwd_ex with that per-wait budget."""
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need("fa_bwd", name, t, _BF16, (B, H, N, d))
    _need("fa_bwd", "lse", lse, _F32, (B, H, N))
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _need("fa_bwd", name, t, (dq.dtype,) if dq.dtype in _OUT else _OUT, (B, H, N, d))
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N), dtype=torch.uint8, device=q.device)
    _need("fa_bwd", "workspace", workspace, _U8)
    ws_bytes = workspace.numel() * workspace.element_size()
    grad_fp32 = int(dq.dtype == torch.float32)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d,
            float(scale), int(bool(causal)), grad_fp32, _ptr(workspace), ws_bytes, _stream(stream))
    if wait_budget_cycles:
        opts = FaBwdOpts(int(wait_budget_cycles))
        _check(lib().fa_bwd_ex(*args, ctypes.byref(opts)), "fa_bwd_ex")
    else:
        _check(lib().fa_bwd(*args), "fa_bwd")


def fa_decode_workspace_bytes(B: int, H: int, L: int, d: int, chunk: int = 128, splits: int = 0) -> int:
    return int(lib().fa_decode_workspace_bytes(B, H, L, d, chunk, splits))


def fa_decode_splitkv(q, k, v, o, lse, scale: float, workspace, chunk: int = 128, splits: int = 0, stream=None,
                      wait_budget_cycles: int = 0):
    """Split-KV decode: q [B, H, d], k/v [B, H, L, d], o [B, H, d] bf16 or fp32 (from its dtype),
    lse [B, H]; workspace a uint8 CUDA tensor (fa_decode_splitkv_ex)."""
    B, H, L, d = k.shape
    _need("fa_decode_splitkv", "q", q, _BF16, (B, H, d))
    _need("fa_decode_splitkv", "k", k, _BF16)
    _need("fa_decode_splitkv", "v", v, _BF16, (B, H, L, d))
    _need("fa_decode_splitkv", "o", o, _OUT, (B, H, d))
    _need("fa_decode_splitkv", "lse", lse, _F32, (B, H))
    if workspace is not None:
        _need("fa_decode_splitkv", "workspace", workspace, _U8)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    opts = FaDecodeOpts(int(o.dtype == torch.float32), int(wait_budget_cycles))
    st = lib().fa_decode_splitkv_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d, float(scale), chunk,
                                    splits, _ptr(workspace), ws_bytes, _stream(stream), ctypes.byref(opts))
    _check(st, "fa_decode_splitkv_ex")


def fa_decode_splitkv_noalloc(q, k, v, o, lse, scale: float, chunk: int = 128, splits: int = 0, stream=None):
    """fa_decode_splitkv without a workspace, for callers that cannot allocate device memory.

    The partials go to a fixed 8 MiB device array inside the library; with
    splits=0 the split count is lowered until they fit, an explicit count that
    does not fit raises FattnError(FA_ERR_WORKSPACE).  Calls that overlap on the
    GPU share that array and race: keep them on one stream.
    """
    B, H, L, d = k.shape
    _need("fa_decode_splitkv_noalloc", "q", q, _BF16, (B, H, d))
    _need("fa_decode_splitkv_noalloc", "k", k, _BF16)
    _need("fa_decode_splitkv_noalloc", "v", v, _BF16, (B, H, L, d))
    _need("fa_decode_splitkv_noalloc", "o", o, _BF16, (B, H, d))
    _need("fa_decode_splitkv_noalloc", "lse", lse, _F32, (B, H))
    st = lib().fa_decode_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, L, d, float(scale),
                                         chunk, splits, _stream(stream))
    _check(st, "fa_decode_splitkv_noalloc")


def fa_decode_paged_workspace_bytes(B: int, H: int, max_seq_len: int, d: int, page_size: int, max_pages: int,
                                    splits: int = 0) -> int:
    return int(lib().fa_decode_paged_workspace_bytes(B, H, max_seq_len, d, page_size, max_pages, splits))


def fa_decode_paged(q, k_pages, v_pages, block_table, seq_lens, o, lse, scale: float, max_seq_len: int,
                    workspace=None, splits: int = 0, stream=None, wait_budget_cycles: int = 0):
    """Split-KV decode over a paged cache: q [B, H, d]; k_pages/v_pages [P, H, page_size, d];
    block_table [B, max_pages] int32; seq_lens [B] int32; o [B, H, d] bf16 or fp32 (from its
    dtype); lse [B, H] fp32 (fa_decode_paged_ex)."""
    B, H, d = q.shape
    P, _, page_size, _ = k_pages.shape
    max_pages = block_table.shape[1]
    _need("fa_decode_paged", "q", q, _BF16, (B, H, d))
    _need("fa_decode_paged", "k_pages", k_pages, _BF16, (P, H, page_size, d))
    _need("fa_decode_paged", "v_pages", v_pages, _BF16, (P, H, page_size, d))
    _need("fa_decode_paged", "block_table", block_table, _I32, (B, max_pages))
    _need("fa_decode_paged", "seq_lens", seq_lens, _I32, (B,))
    _need("fa_decode_paged", "o", o, _OUT, (B, H, d))
    _need("fa_decode_paged", "lse", lse, _F32, (B, H))
    if workspace is None:
        workspace = torch.empty(fa_decode_paged_workspace_bytes(B, H, max_seq_len, d, page_size, max_pages, splits),
                                dtype=torch.uint8, device=q.device)
    _need("fa_decode_paged", "workspace", workspace, _U8)
    ws_bytes = workspace.numel() * workspace.element_size()
    opts = FaDecodeOpts(int(o.dtype == torch.float32), int(wait_budget_cycles))
    st = lib().fa_decode_paged_ex(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), _ptr(o),
                                  _ptr(lse), B, H, d, page_size, max_pages, P, max_seq_len, float(scale), splits,
                                  _ptr(workspace), ws_bytes, _stream(stream), ctypes.byref(opts))
    _check(st, "fa_decode_paged_ex")


def fa_combine(u_part, m_part, l_part, o, lse, stream=None):
    """Merge partials: u_part [R, S, d], m_part/l_part [R, S] fp32 -> o [R, d] bf16 or fp32 (from its
    dtype; fa_combine_ex), lse [R] fp32."""
    R, S, d = u_part.shape
    _need("fa_combine", "u_part", u_part, _F32, (R, S, d))
    _need("fa_combine", "m_part", m_part, _F32, (R, S))
    _need("fa_combine", "l_part", l_part, _F32, (R, S))
    _need("fa_combine", "o", o, _OUT, (R, d))
    _need("fa_combine", "lse", lse, _F32, (R,))
    st = lib().fa_combine_ex(_ptr(u_part), _ptr(m_part), _ptr(l_part), _ptr(o), _ptr(lse), R, S, d,
                             int(o.dtype == torch.float32), _stream(stream))
    _check(st, "fa_combine_ex")


def fa_get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the kernels' status; raises on a timeout."""
    st = lib().fa_get_status(_stream(stream))
    _check(st, "fa_get_status")
    return st
