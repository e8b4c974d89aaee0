"""Python binding of the C ABI in ``include/pagedattn.h``.

Argument marshalling only: shapes are read off torch tensors, pointers and the
current CUDA stream are passed through ctypes, and a non-zero ``pa_status``
raises :class:`PaError`.  Every step of the computation runs in the CUDA
library ``libpagedattn.so``; there is no fallback path.  torch is used for
device memory and streams only.

Dtypes follow the pages (AstrAI commit 398e8a3, tests/inference/test_cache.py):
bf16 activations and KV buffers, int32 page-table / request-row / location
indices; the fp8 entry points take e4m3 caches (uint8 or float8_e4m3fn
tensors) with fp32 [n_layers, n_kv_heads] scales.  Other dtypes are rejected
here, before any launch.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

PA_OK = 0
STATUS = {0: "PA_OK", 1: "PA_ERR_NULL", 2: "PA_ERR_SHAPE", 3: "PA_ERR_ALIGN", 4: "PA_ERR_UNSUPPORTED",
          5: "PA_ERR_WORKSPACE", 6: "PA_ERR_CUDA", 7: "PA_ERR_DEVICE_INDEX"}
DEVERR_SLOT, DEVERR_ROW, DEVERR_LEN, DEVERR_POS, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
OVERLAP_OFF, OVERLAP_SAFE, OVERLAP_EARLY_METADATA, OVERLAP_EARLY_KV = 0, 1, 2, 3


class PaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


class CascadeCaps(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int), ("max_groups", ctypes.c_int), ("max_group_size", ctypes.c_int),
                ("max_splits", ctypes.c_int)]


class KvShape(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("size", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int)]


EXPORTS = ["pa_status_string", "pa_decode_workspace_bytes", "pa_prefill_workspace_bytes",
           "pa_workspace_init", "pa_get_error", "pa_get_error_word", "pa_kv_store", "pa_rope_packed",
           "pa_paged_decode_attn", "pa_paged_prefill_attn", "pa_paged_decode_attn_noalloc",
           "pa_set_launch_overlap", "pa_get_launch_overlap", "pa_decode_step",
           "pa_paged_prefill_attn_last", "pa_dense_prefill_attn", "pa_cascade_workspace_bytes",
           "pa_paged_decode_attn_cascade", "pa_kv_store_fp8", "pa_paged_decode_attn_fp8",
           "pa_paged_prefill_attn_fp8", "pa_set_wait_timeout_ns", "pa_get_wait_timeout_ns"]

_lib = None


def lib():
    """Load libpagedattn.so (built by ``paged_kv_cache_188_gb300.build``); fail loudly if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run paged_kv_cache_188_gb300.build.build() first "
                           "(the CUDA library is required; there is no CPU path)")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    L.pa_status_string.argtypes = [i32]
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.pa_decode_workspace_bytes.restype = sz
    L.pa_prefill_workspace_bytes.argtypes = []
    L.pa_prefill_workspace_bytes.restype = sz
    L.pa_workspace_init.argtypes = [P, sz, P]
    L.pa_get_error.argtypes = [P, P, P]
    L.pa_get_error_word.argtypes = [P, P, P]
    L.pa_kv_store.argtypes = [P, P, KvShape, i32, P, P, P, i32, P, P]
    L.pa_rope_packed.argtypes = [P, i32, P, i32, i32, P, i32, P, P, i32, P, P]
    L.pa_paged_decode_attn.argtypes = [P, i32, i32, P, P, KvShape, i32, P, i32, i32, P, P, f32, P, sz, i32,
                                       P, P]
    L.pa_paged_prefill_attn.argtypes = [P, i32, i32, P, P, KvShape, i32, P, P, i32, P, i32, i32, P, f32, P,
                                        sz, P, P]
    L.pa_paged_decode_attn_noalloc.argtypes = [P, i32, i32, P, P, KvShape, i32, P, i32, i32, P, P, f32, i32, P,
                                               P, P]
    L.pa_decode_step.argtypes = [P, P, P, i32, i32, P, P, P, i32, P, P, KvShape, i32, P, P, i32, i32, P, P, f32,
                                 P, sz, i32, P, P]
    L.pa_paged_prefill_attn_last.argtypes = [P, i32, i32, P, P, KvShape, i32, P, P, i32, P, i32, i32, P, f32, P,
                                             sz, P, P, P]
    L.pa_dense_prefill_attn.argtypes = [P, i32, i32, P, P, i32, i32, P, i32, f32, P, sz, P, P, P]
    L.pa_cascade_workspace_bytes.argtypes = [CascadeCaps, i32, i32, i32]
    L.pa_paged_decode_attn_cascade.argtypes = [P, i32, i32, P, P, KvShape, i32, P, i32, i32, P, P, P, P, P, i32,
                                               CascadeCaps, f32, P, sz, P, P]
    L.pa_kv_store_fp8.argtypes = [P, P, KvShape, i32, P, P, P, i32, P, P, P, P]
    L.pa_paged_decode_attn_fp8.argtypes = [P, i32, i32, P, P, KvShape, i32, P, i32, i32, P, P, f32, P, P, P, sz,
                                           i32, P, P]
    L.pa_paged_prefill_attn_fp8.argtypes = [P, i32, i32, P, P, KvShape, i32, P, P, i32, P, i32, i32, P, f32, P, P,
                                            P, sz, P, P]
    L.pa_set_launch_overlap.argtypes = [i32]
    L.pa_get_launch_overlap.argtypes = []
    L.pa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.pa_get_wait_timeout_ns.argtypes = []
    for name in EXPORTS[3:]:
        getattr(L, name).restype = i32
    L.pa_cascade_workspace_bytes.restype = sz
    L.pa_set_wait_timeout_ns.restype = None
    L.pa_get_wait_timeout_ns.restype = ctypes.c_uint64
    _lib = L
    return L


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _ok(fn, rc):
    if rc != PA_OK:
        raise PaError(fn, rc)


def _kv_shape(k_buf, v_buf):
    _need(k_buf, torch.bfloat16, "k_buf", 4)
    _need(v_buf, torch.bfloat16, "v_buf", 4)
    if k_buf.shape != v_buf.shape:
        raise ValueError("k_buf and v_buf shapes differ")
    return KvShape(*k_buf.shape)


FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _kv_shape_fp8(k_buf, v_buf, k_scale, v_scale):
    """An e4m3 cache: uint8 (or float8_e4m3fn) [n_layers, size, Hkv, D] buffers
    and fp32 [n_layers, Hkv] scales."""
    for t, name in ((k_buf, "k_buf"), (v_buf, "v_buf")):
        if t.dtype not in FP8_DTYPES:
            raise TypeError(f"{name} must be uint8 or float8_e4m3fn, got {t.dtype}")
        _need(t, t.dtype, name, 4)
    if k_buf.shape != v_buf.shape:
        raise ValueError("k_buf and v_buf shapes differ")
    _need(k_scale, torch.float32, "k_scale", 2)
    _need(v_scale, torch.float32, "v_scale", 2)
    if tuple(k_scale.shape) != tuple(k_buf.shape[:1] + k_buf.shape[2:3]) or v_scale.shape != k_scale.shape:
        raise ValueError("k_scale / v_scale must be [n_layers, n_kv_heads]")
    return KvShape(*k_buf.shape)


def pa_set_launch_overlap(mode):
    """Process-wide launch overlap (OVERLAP_OFF / OVERLAP_SAFE / OVERLAP_EARLY_METADATA / OVERLAP_EARLY_KV)."""
    _ok("pa_set_launch_overlap", lib().pa_set_launch_overlap(int(mode)))


def pa_get_launch_overlap():
    return int(lib().pa_get_launch_overlap())


def pa_decode_workspace_bytes(max_batch, n_q_heads, n_kv_heads, head_dim, max_splits):
    return int(lib().pa_decode_workspace_bytes(max_batch, n_q_heads, n_kv_heads, head_dim, max_splits))


def pa_prefill_workspace_bytes():
    return int(lib().pa_prefill_workspace_bytes())


def alloc_workspace(nbytes, device="cuda"):
    """A zero-initialised, 256-byte aligned workspace (torch's allocator aligns to 512 B)."""
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def pa_workspace_init(workspace, stream=None):
    _ok("pa_workspace_init", lib().pa_workspace_init(_p(workspace), workspace.numel(), _stream(stream)))


def pa_get_error(workspace, stream=None):
    """Device error word of a workspace (synchronises the stream)."""
    v = ctypes.c_int32(0)
    rc = lib().pa_get_error(_p(workspace), ctypes.byref(v), _stream(stream))
    if rc not in (PA_OK, 7):
        raise PaError("pa_get_error", rc)
    return int(v.value)


def pa_get_error_word(error_word, stream=None):
    v = ctypes.c_int32(0)
    rc = lib().pa_get_error_word(_p(error_word), ctypes.byref(v), _stream(stream))
    if rc not in (PA_OK, 7):
        raise PaError("pa_get_error_word", rc)
    return int(v.value)


def pa_kv_store(k_buf, v_buf, layer_id, k_new, v_new, loc, error_word=None, stream=None):
    s = _kv_shape(k_buf, v_buf)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(loc, torch.int32, "loc", 1)
    T = loc.numel()
    if tuple(k_new.shape) != (T, s.n_kv_heads, s.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [n_tokens, n_kv_heads, head_dim]")
    if error_word is not None:
        _need(error_word, torch.int32, "error_word")
    _ok("pa_kv_store", lib().pa_kv_store(_p(k_buf), _p(v_buf), s, layer_id, _p(k_new), _p(v_new), _p(loc), T,
                                         _p(error_word), _stream(stream)))


def pa_kv_store_fp8(k_buf, v_buf, layer_id, k_new, v_new, loc, k_scale, v_scale, error_word=None, stream=None):
    """Quantising KV store into an e4m3 cache (bf16 rows divided by their
    (layer, kv head) scale, rounded to e4m3)."""
    s = _kv_shape_fp8(k_buf, v_buf, k_scale, v_scale)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(loc, torch.int32, "loc", 1)
    T = loc.numel()
    if tuple(k_new.shape) != (T, s.n_kv_heads, s.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [n_tokens, n_kv_heads, head_dim]")
    if error_word is not None:
        _need(error_word, torch.int32, "error_word")
    _ok("pa_kv_store_fp8", lib().pa_kv_store_fp8(_p(k_buf), _p(v_buf), s, layer_id, _p(k_new), _p(v_new), _p(loc),
                                                 T, _p(k_scale), _p(v_scale), _p(error_word), _stream(stream)))


def pa_rope_packed(q, k, positions, cos_tab, sin_tab, error_word=None, stream=None):
    _need(q, torch.bfloat16, "q", 3)
    _need(positions, torch.int32, "positions", 1)
    _need(cos_tab, torch.float32, "cos_tab", 2)
    _need(sin_tab, torch.float32, "sin_tab", 2)
    T, Hq, D = q.shape
    Hkv = 0
    if k is not None:
        _need(k, torch.bfloat16, "k", 3)
        if k.shape[0] != T or k.shape[2] != D:
            raise ValueError("k must be [n_tokens, n_kv_heads, head_dim]")
        Hkv = k.shape[1]
    if positions.numel() != T or cos_tab.shape != sin_tab.shape or cos_tab.shape[1] != D // 2:
        raise ValueError("positions [T] and cos/sin tables [max_pos, head_dim/2] expected")
    if error_word is not None:
        _need(error_word, torch.int32, "error_word")
    _ok("pa_rope_packed", lib().pa_rope_packed(_p(q), Hq, _p(k), Hkv, D, _p(positions), T, _p(cos_tab),
                                               _p(sin_tab), cos_tab.shape[0], _p(error_word), _stream(stream)))


def pa_paged_decode_attn(q, k_buf, v_buf, layer_id, req_to_token, req_pool_indices, seq_lens, scale,
                         workspace, max_splits, out, stream=None):
    s = _kv_shape(k_buf, v_buf)
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(req_to_token, torch.int32, "req_to_token", 2)
    _need(req_pool_indices, torch.int32, "req_pool_indices", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(workspace, torch.uint8, "workspace")
    B, Hq, D = q.shape
    if out.shape != q.shape or D != s.head_dim or req_pool_indices.numel() != B or seq_lens.numel() != B:
        raise ValueError("q/out [batch, n_q_heads, head_dim], req_pool_indices/seq_lens [batch] expected")
    _ok("pa_paged_decode_attn", lib().pa_paged_decode_attn(
        _p(q), B, Hq, _p(k_buf), _p(v_buf), s, layer_id, _p(req_to_token), req_to_token.shape[0],
        req_to_token.shape[1], _p(req_pool_indices), _p(seq_lens), float(scale), _p(workspace),
        workspace.numel(), max_splits, _p(out), _stream(stream)))


def pa_paged_decode_attn_fp8(q, k_buf, v_buf, layer_id, req_to_token, req_pool_indices, seq_lens, scale,
                             k_scale, v_scale, workspace, max_splits, out, stream=None):
    """Decode attention over an e4m3 cache with per-(layer, kv head) scales."""
    s = _kv_shape_fp8(k_buf, v_buf, k_scale, v_scale)
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(req_to_token, torch.int32, "req_to_token", 2)
    _need(req_pool_indices, torch.int32, "req_pool_indices", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(workspace, torch.uint8, "workspace")
    B, Hq, D = q.shape
    if out.shape != q.shape or D != s.head_dim or req_pool_indices.numel() != B or seq_lens.numel() != B:
        raise ValueError("q/out [batch, n_q_heads, head_dim], req_pool_indices/seq_lens [batch] expected")
    _ok("pa_paged_decode_attn_fp8", lib().pa_paged_decode_attn_fp8(
        _p(q), B, Hq, _p(k_buf), _p(v_buf), s, layer_id, _p(req_to_token), req_to_token.shape[0],
        req_to_token.shape[1], _p(req_pool_indices), _p(seq_lens), float(scale), _p(k_scale), _p(v_scale),
        _p(workspace), workspace.numel(), max_splits, _p(out), _stream(stream)))


def pa_decode_step(q, k_new, v_new, positions, cos_tab, sin_tab, k_buf, v_buf, layer_id, loc, req_to_token,
                   req_pool_indices, seq_lens, scale, workspace, max_splits, out, stream=None):
    """RoPE + KV store + decode attention of one layer in one launch (q, k_new only read)."""
    s = _kv_shape(k_buf, v_buf)
    _need(q, torch.bfloat16, "q", 3)
    _need(k_new, torch.bfloat16, "k_new", 3)
    _need(v_new, torch.bfloat16, "v_new", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(positions, torch.int32, "positions", 1)
    _need(loc, torch.int32, "loc", 1)
    _need(cos_tab, torch.float32, "cos_tab", 2)
    _need(sin_tab, torch.float32, "sin_tab", 2)
    _need(req_to_token, torch.int32, "req_to_token", 2)
    _need(req_pool_indices, torch.int32, "req_pool_indices", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(workspace, torch.uint8, "workspace")
    B, Hq, D = q.shape
    if (out.shape != q.shape or D != s.head_dim or k_new.shape != (B, s.n_kv_heads, D) or v_new.shape != k_new.shape
            or positions.numel() != B or loc.numel() != B or req_pool_indices.numel() != B or seq_lens.numel() != B
            or cos_tab.shape != sin_tab.shape or cos_tab.shape[1] != D // 2):
        raise ValueError("q/out [batch, Hq, D], k_new/v_new [batch, Hkv, D], positions/loc/req_pool_indices/"
                         "seq_lens [batch], cos/sin [max_pos, D/2] expected")
    _ok("pa_decode_step", lib().pa_decode_step(
        _p(q), _p(k_new), _p(v_new), B, Hq, _p(positions), _p(cos_tab), _p(sin_tab), cos_tab.shape[0],
        _p(k_buf), _p(v_buf), s, layer_id, _p(loc), _p(req_to_token), req_to_token.shape[0], req_to_token.shape[1],
        _p(req_pool_indices), _p(seq_lens), float(scale), _p(workspace), workspace.numel(), max_splits, _p(out),
        _stream(stream)))


def pa_paged_decode_attn_noalloc(q, k_buf, v_buf, layer_id, req_to_token, req_pool_indices, seq_lens, scale,
                                 max_splits, out, error_word=None, stream=None):
    """pa_paged_decode_attn with the library's fixed internal scratch instead of a workspace."""
    s = _kv_shape(k_buf, v_buf)
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(req_to_token, torch.int32, "req_to_token", 2)
    _need(req_pool_indices, torch.int32, "req_pool_indices", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    if error_word is not None:
        _need(error_word, torch.int32, "error_word")
    B, Hq, D = q.shape
    if out.shape != q.shape or D != s.head_dim or req_pool_indices.numel() != B or seq_lens.numel() != B:
        raise ValueError("q/out [batch, n_q_heads, head_dim], req_pool_indices/seq_lens [batch] expected")
    _ok("pa_paged_decode_attn_noalloc", lib().pa_paged_decode_attn_noalloc(
        _p(q), B, Hq, _p(k_buf), _p(v_buf), s, layer_id, _p(req_to_token), req_to_token.shape[0],
        req_to_token.shape[1], _p(req_pool_indices), _p(seq_lens), float(scale), max_splits, _p(out),
        _p(error_word), _stream(stream)))


WAIT_TIMEOUT_DEFAULT_NS = 2_000_000_000


def pa_set_wait_timeout_ns(ns):
    """Time limit of the kernels' bounded pipeline waits; 0 makes every wait
    give up at once (a test hook for the abort path)."""
    lib().pa_set_wait_timeout_ns(int(ns))


def pa_get_wait_timeout_ns():
    return int(lib().pa_get_wait_timeout_ns())


def pa_paged_prefill_attn_fp8(q, k_buf, v_buf, layer_id, qo_indptr, kv_indptr, req_to_token, req_pool_indices,
                              scale, k_scale, v_scale, workspace, out, stream=None):
    """Ragged causal prefill over an e4m3 cache with per-(layer, kv head) scales."""
    s = _kv_shape_fp8(k_buf, v_buf, k_scale, v_scale)
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(qo_indptr, torch.int32, "qo_indptr", 1)
    _need(kv_indptr, torch.int32, "kv_indptr", 1)
    _need(req_to_token, torch.int32, "req_to_token", 2)
    _need(req_pool_indices, torch.int32, "req_pool_indices", 1)
    _need(workspace, torch.uint8, "workspace")
    T, Hq, D = q.shape
    R = qo_indptr.numel() - 1
    if out.shape != q.shape or D != s.head_dim or kv_indptr.numel() != R + 1 or req_pool_indices.numel() != R:
        raise ValueError("q/out [T, Hq, D], qo/kv_indptr [R+1], req_pool_indices [R] expected")
    _ok("pa_paged_prefill_attn_fp8", lib().pa_paged_prefill_attn_fp8(
        _p(q), T, Hq, _p(k_buf), _p(v_buf), s, layer_id, _p(qo_indptr), _p(kv_indptr), R, _p(req_to_token),
        req_to_token.shape[0], req_to_token.shape[1], _p(req_pool_indices), float(scale), _p(k_scale), _p(v_scale),
        _p(workspace), workspace.numel(), _p(out), _stream(stream)))


def pa_paged_prefill_attn(q, k_buf, v_buf, layer_id, qo_indptr, kv_indptr, req_to_token, req_pool_indices,
                          scale, workspace, out, stream=None, last_out=None):
    """Ragged causal prefill over the paged cache; with ``last_out`` ([R, Hq, D])
    each request's last row is also gathered there by the same kernel."""
    s = _kv_shape(k_buf, v_buf)
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(qo_indptr, torch.int32, "qo_indptr", 1)
    _need(kv_indptr, torch.int32, "kv_indptr", 1)
    _need(req_to_token, torch.int32, "req_to_token", 2)
    _need(req_pool_indices, torch.int32, "req_pool_indices", 1)
    _need(workspace, torch.uint8, "workspace")
    T, Hq, D = q.shape
    R = qo_indptr.numel() - 1
    if out.shape != q.shape or D != s.head_dim or kv_indptr.numel() != R + 1 or req_pool_indices.numel() != R:
        raise ValueError("q/out [T, n_q_heads, head_dim], indptrs [R+1], req_pool_indices [R] expected")
    args = [_p(q), T, Hq, _p(k_buf), _p(v_buf), s, layer_id, _p(qo_indptr), _p(kv_indptr), R, _p(req_to_token),
            req_to_token.shape[0], req_to_token.shape[1], _p(req_pool_indices), float(scale), _p(workspace),
            workspace.numel(), _p(out)]
    if last_out is None:
        _ok("pa_paged_prefill_attn", lib().pa_paged_prefill_attn(*args, _stream(stream)))
    else:
        _need(last_out, torch.bfloat16, "last_out", 3)
        if last_out.shape != (R, Hq, D):
            raise ValueError("last_out [R, n_q_heads, head_dim] expected")
        _ok("pa_paged_prefill_attn_last", lib().pa_paged_prefill_attn_last(*args, _p(last_out), _stream(stream)))


def pa_dense_prefill_attn(q, k, v, qo_indptr, scale, workspace, out, last_out=None, stream=None):
    """Causal prefill of packed prompts with no cached prefix: K/V are the new
    tokens' packed rows [T, Hkv, D], no page table."""
    _need(q, torch.bfloat16, "q", 3)
    _need(k, torch.bfloat16, "k", 3)
    _need(v, torch.bfloat16, "v", 3)
    _need(out, torch.bfloat16, "out", 3)
    _need(qo_indptr, torch.int32, "qo_indptr", 1)
    _need(workspace, torch.uint8, "workspace")
    T, Hq, D = q.shape
    R = qo_indptr.numel() - 1
    if out.shape != q.shape or k.shape != v.shape or k.shape[0] != T or k.shape[2] != D:
        raise ValueError("q/out [T, Hq, D], k/v [T, Hkv, D] expected")
    if last_out is not None:
        _need(last_out, torch.bfloat16, "last_out", 3)
        if last_out.shape != (R, Hq, D):
            raise ValueError("last_out [R, n_q_heads, head_dim] expected")
    _ok("pa_dense_prefill_attn", lib().pa_dense_prefill_attn(
        _p(q), T, Hq, _p(k), _p(v), k.shape[1], D, _p(qo_indptr), R, float(scale), _p(workspace), workspace.numel(),
        _p(out), _p(last_out), _stream(stream)))


def pa_cascade_workspace_bytes(max_batch, max_groups, max_group_size, max_splits, n_q_heads, n_kv_heads, head_dim):
    return int(lib().pa_cascade_workspace_bytes(CascadeCaps(max_batch, max_groups, max_group_size, max_splits),
                                                n_q_heads, n_kv_heads, head_dim))


def pa_paged_decode_attn_cascade(q, k_buf, v_buf, layer_id, req_to_token, req_pool_indices, seq_lens, group_indptr,
                                 group_reqs, group_prefix, scale, workspace, caps, out, stream=None):
    """Decode attention with shared prefixes read once per chunk of group members.

    ``caps`` = (max_batch, max_groups, max_group_size, max_splits): the same for
    every call on one workspace (it fixes the workspace layout)."""
    s = _kv_shape(k_buf, v_buf)
    _need(q, torch.bfloat16, "q", 3)
    _need(out, torch.bfloat16, "out", 3)
    for t, n in ((req_to_token, "req_to_token"), (req_pool_indices, "req_pool_indices"), (seq_lens, "seq_lens"),
                 (group_indptr, "group_indptr"), (group_reqs, "group_reqs"), (group_prefix, "group_prefix")):
        _need(t, torch.int32, n)
    _need(workspace, torch.uint8, "workspace")
    B, Hq, D = q.shape
    n_groups = group_indptr.numel() - 1
    if out.shape != q.shape or D != s.head_dim or group_prefix.numel() != n_groups:
        raise ValueError("q/out [batch, Hq, D], group_indptr [n_groups + 1], group_prefix [n_groups] expected")
    _ok("pa_paged_decode_attn_cascade", lib().pa_paged_decode_attn_cascade(
        _p(q), B, Hq, _p(k_buf), _p(v_buf), s, layer_id, _p(req_to_token), req_to_token.shape[0],
        req_to_token.shape[1], _p(req_pool_indices), _p(seq_lens), _p(group_indptr), _p(group_reqs),
        _p(group_prefix), n_groups, CascadeCaps(*caps), float(scale), _p(workspace), workspace.numel(), _p(out),
        _stream(stream)))
