"""ctypes binding of libattn_sm103.so (include/attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  If the library has not been built, the first call raises -- there
is no fallback of any kind.
"""
import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libattn_sm103.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "attn.h")

ATTN_OK = 0
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_DEVICE_ARG = 6
STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_MISALIGNED",
    4: "ATTN_ERR_LAUNCH", 5: "ATTN_ERR_TIMEOUT", 6: "ATTN_ERR_DEVICE_ARG", 7: "ATTN_ERR_WORKSPACE",
}

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s failed: %s (%s)" % (what, STATUS_NAMES.get(code, code), status_string(code)))


def declared_functions():
    """Names of the functions include/attn.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:ATTN_API\s+)?(?:const\s+)?\w+\**\s+\**(attn_\w+)\s*\(", text, flags=re.M)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("CUDA attention library not built (%s); run __graft_entry__.build()" % LIB_PATH)
        _lib = _open(LIB_PATH)
    return _lib


_variants = {}


def variant_lib(name):
    """A build variant of the library (same interface; see build.VARIANTS),
    built on first use.  Pass it as ``library=`` to the calls below."""
    if name not in _variants:
        from . import build as _build
        _variants[name] = _open(_build.build_variant(name))
    return _variants[name]


def _open(path):
    """Loads one build of the library and declares its C signatures."""
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.restype = i
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.attn_fwd_window.restype = i
    L.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp]
    L.attn_fwd_kvcache.restype = i
    L.attn_fwd_kvcache.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, i, i, f, vp]
    L.attn_splitkv_workspace_size.restype = sz
    L.attn_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    L.attn_fwd_splitkv.restype = i
    L.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    L.attn_fwd_splitkv_paged.restype = i
    L.attn_fwd_splitkv_paged.argtypes = [vp, vp, vp, vp, i, i, i, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    L.attn_fwd_splitkv_noalloc.restype = i
    L.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, f, i, vp]
    L.attn_get_device_status.restype = i
    L.attn_get_device_status.argtypes = [vp]
    L.attn_selftest_wait_timeout.restype = i
    L.attn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_status_string.argtypes = [i]
    L.attn_selftest_exp2_poly.restype = i
    L.attn_selftest_exp2_poly.argtypes = [vp, vp, ctypes.c_longlong, vp]
    L.attn_probe_read_bandwidth.restype = i
    L.attn_probe_read_bandwidth.argtypes = [vp, sz, vp, vp]
    return L


def status_string(code: int) -> str:
    return lib().attn_status_string(int(code)).decode()


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_bf16(name, t, shape):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be a contiguous CUDA bf16 tensor of shape %s (got %s %s %s)"
                         % (name, tuple(shape), t.dtype, tuple(t.shape), t.device))


# --------------------------------------------------------------------------- raw entry points
def _check_prefill(q, k, v, o, lse):
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    _check_bf16("q", q, (B, Nq, Hq, d))
    _check_bf16("k", k, (B, Nk, Hkv, d))
    _check_bf16("v", v, (B, Nk, Hkv, d))
    _check_bf16("o", o, (B, Nq, Hq, d))
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of shape %s" % ((B, Hq, Nq),))
    return B, Hq, Hkv, Nq, Nk, d


def _window(window):
    """None or (left, right); a negative side is unbounded."""
    if window is None:
        return -1, -1
    wl, wr = (int(x) for x in window)
    return wl, wr


def attn_fwd(q, k, v, o, lse, causal, scale, stream=None, library=None):
    """Same contract as the C call: writes o [B,Nq,Hq,d] and lse [B,Hq,Nq]. Returns the status.
    library: a build variant from variant_lib(), else the default build."""
    B, Hq, Hkv, Nq, Nk, d = _check_prefill(q, k, v, o, lse)
    return (library or lib()).attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                       int(causal), float(scale), _stream_handle(stream))


def attn_fwd_window(q, k, v, o, lse, causal, window, scale, stream=None):
    """attn_fwd with a local window (left, right), aligned bottom-right. Returns the status."""
    B, Hq, Hkv, Nq, Nk, d = _check_prefill(q, k, v, o, lse)
    wl, wr = _window(window)
    return lib().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                 int(causal), wl, wr, float(scale), _stream_handle(stream))


def attn_fwd_kvcache(q, k_cache, v_cache, seqlens, o, lse, causal, scale, stream=None, window=None):
    """Same contract as the C call: q, o [B,Nq,Hq,d]; caches [B,max_seqlen,Hkv,d];
    seqlens int32 [B] on the device; lse [B,Hq,Nq].  Returns the status."""
    B, Nq, Hq, d = q.shape
    max_seqlen, Hkv = k_cache.shape[1], k_cache.shape[2]
    _check_bf16("q", q, (B, Nq, Hq, d))
    _check_bf16("k_cache", k_cache, (B, max_seqlen, Hkv, d))
    _check_bf16("v_cache", v_cache, (B, max_seqlen, Hkv, d))
    _check_bf16("o", o, (B, Nq, Hq, d))
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or tuple(seqlens.shape) != (B,):
        raise ValueError("seqlens must be a CUDA int32 tensor of shape (%d,)" % B)
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor of shape %s" % ((B, Hq, Nq),))
    wl, wr = _window(window)
    return lib().attn_fwd_kvcache(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), max_seqlen, _ptr(o),
                                  _ptr(lse), B, Hq, Hkv, Nq, d, int(causal), wl, wr, float(scale),
                                  _stream_handle(stream))


def forward_kvcache(q, k_cache, v_cache, seqlens, causal, scale, stream=None, window=None):
    """Allocates O and LSE and runs attn_fwd_kvcache. Returns (o, lse)."""
    B, Nq, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    rc = attn_fwd_kvcache(q, k_cache, v_cache, seqlens, o, lse, causal, scale, stream, window)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_kvcache")
    return o, lse


def attn_splitkv_workspace_size(B, Hq, max_seqlen, d, chunk):
    return int(lib().attn_splitkv_workspace_size(B, Hq, max_seqlen, d, chunk))


def attn_fwd_splitkv(q, k_cache, v_cache, seqlens, o, lse, scale, chunk, workspace, stream=None):
    """Same contract as the C call. workspace: a CUDA uint8 tensor. Returns the status."""
    B, _, Hq, d = q.shape
    max_seqlen, Hkv = k_cache.shape[1], k_cache.shape[2]
    _check_bf16("q", q, (B, 1, Hq, d))
    _check_bf16("k_cache", k_cache, (B, max_seqlen, Hkv, d))
    _check_bf16("v_cache", v_cache, (B, max_seqlen, Hkv, d))
    _check_bf16("o", o, (B, 1, Hq, d))
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or tuple(seqlens.shape) != (B,):
        raise ValueError("seqlens must be a CUDA int32 tensor of shape (%d,)" % B)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, Hq, 1):
        raise ValueError("lse must be a CUDA fp32 tensor of shape %s" % ((B, Hq, 1),))
    return lib().attn_fwd_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), max_seqlen,
                                  _ptr(o), _ptr(lse), B, Hq, Hkv, d, float(scale), int(chunk),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))


def attn_fwd_splitkv_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, scale, chunk, workspace, stream=None):
    """Same contract as the C call: k_pages, v_pages [num_pages, page_size, Hkv, d];
    block_table int32 [B, max_blocks] on the device.  Returns the status."""
    B, _, Hq, d = q.shape
    num_pages, page_size, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    max_blocks = block_table.shape[1]
    _check_bf16("q", q, (B, 1, Hq, d))
    _check_bf16("k_pages", k_pages, (num_pages, page_size, Hkv, d))
    _check_bf16("v_pages", v_pages, (num_pages, page_size, Hkv, d))
    _check_bf16("o", o, (B, 1, Hq, d))
    if block_table.dtype != torch.int32 or not block_table.is_cuda or not block_table.is_contiguous() \
            or tuple(block_table.shape) != (B, max_blocks):
        raise ValueError("block_table must be a contiguous CUDA int32 tensor of shape (%d, max_blocks)" % B)
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or tuple(seqlens.shape) != (B,):
        raise ValueError("seqlens must be a CUDA int32 tensor of shape (%d,)" % B)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, Hq, 1):
        raise ValueError("lse must be a CUDA fp32 tensor of shape %s" % ((B, Hq, 1),))
    return lib().attn_fwd_splitkv_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), max_blocks,
                                        page_size, num_pages, _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv, d,
                                        float(scale), int(chunk), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream_handle(stream))


def attn_fwd_splitkv_noalloc(q, k_cache, v_cache, seqlens, o, lse, scale, chunk, stream=None):
    """attn_fwd_splitkv without a workspace: the library's fixed device scratch
    holds the partials, so nothing is allocated (for callers that cannot
    allocate device memory).  Returns the status."""
    B, _, Hq, d = q.shape
    max_seqlen, Hkv = k_cache.shape[1], k_cache.shape[2]
    _check_bf16("q", q, (B, 1, Hq, d))
    _check_bf16("k_cache", k_cache, (B, max_seqlen, Hkv, d))
    _check_bf16("v_cache", v_cache, (B, max_seqlen, Hkv, d))
    _check_bf16("o", o, (B, 1, Hq, d))
    if seqlens.dtype != torch.int32 or not seqlens.is_cuda or tuple(seqlens.shape) != (B,):
        raise ValueError("seqlens must be a CUDA int32 tensor of shape (%d,)" % B)
    if lse.dtype != torch.float32 or not lse.is_cuda or tuple(lse.shape) != (B, Hq, 1):
        raise ValueError("lse must be a CUDA fp32 tensor of shape %s" % ((B, Hq, 1),))
    return lib().attn_fwd_splitkv_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), max_seqlen,
                                          _ptr(o), _ptr(lse), B, Hq, Hkv, d, float(scale), int(chunk),
                                          _stream_handle(stream))


def attn_get_device_status(stream=None):
    return lib().attn_get_device_status(_stream_handle(stream))


def attn_selftest_exp2_poly(x, y, stream=None):
    """y = 2^x by the library's software exp2 (float32 CUDA tensors of one size). Returns the status."""
    for name, t in (("x", x), ("y", y)):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA float32 tensor" % name)
    if x.numel() != y.numel():
        raise ValueError("x and y differ in size")
    return lib().attn_selftest_exp2_poly(_ptr(x), _ptr(y), x.numel(), _stream_handle(stream))


def attn_probe_read_bandwidth(buf, sink, stream=None):
    """One streaming read of the CUDA tensor buf (its bytes; see the C call);
    sink: a CUDA int64 tensor of one element.  Returns the status."""
    if not buf.is_cuda or not buf.is_contiguous() or sink.dtype != torch.int64 or not sink.is_cuda:
        raise ValueError("buf must be a contiguous CUDA tensor and sink a CUDA int64 tensor")
    return lib().attn_probe_read_bandwidth(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                           _stream_handle(stream))


def attn_selftest_wait_timeout(limit_ns, stream=None):
    """Launches the bounded-wait self-test kernel; its timeout shows in attn_get_device_status."""
    return lib().attn_selftest_wait_timeout(int(limit_ns), _stream_handle(stream))


# --------------------------------------------------------------------------- convenience wrappers
def forward(q, k, v, causal, scale, stream=None, library=None):
    """Allocates O and LSE with torch on q's device and runs attn_fwd. Returns (o, lse)."""
    B, Nq, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    rc = attn_fwd(q, k, v, o, lse, causal, scale, stream, library)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd")
    return o, lse


def forward_window(q, k, v, causal, window, scale, stream=None):
    """Allocates O and LSE and runs attn_fwd_window. Returns (o, lse)."""
    B, Nq, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    rc = attn_fwd_window(q, k, v, o, lse, causal, window, scale, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_window")
    return o, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, scale, chunk=1024, workspace=None, stream=None):
    """Allocates O, LSE (and the workspace unless given) and runs attn_fwd_splitkv_paged."""
    B, _, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = attn_splitkv_workspace_size(B, Hq, block_table.shape[1] * k_pages.shape[1], d, chunk)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    rc = attn_fwd_splitkv_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, scale, chunk, workspace, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv_paged")
    return o, lse


def decode(q, k_cache, v_cache, seqlens, scale, chunk=1024, workspace=None, stream=None):
    """Allocates O, LSE (and the workspace unless given) and runs attn_fwd_splitkv."""
    B, _, Hq, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = attn_splitkv_workspace_size(B, Hq, k_cache.shape[1], d, chunk)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
    rc = attn_fwd_splitkv(q, k_cache, v_cache, seqlens, o, lse, scale, chunk, workspace, stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv")
    return o, lse
