"""Float64 CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is the checker that the CUDA library is
compared against: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import it.  The product package
(``paged_kv_cache_188_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, single-threaded),
compiled with gcc into ``liboracle.so`` next to this file.  This module only
marshals numpy arrays through ctypes.  Every function states the definition it
computes and the page passage it follows in ``oracle.c``.

bf16 tensors are passed as ``numpy.uint16`` arrays of bit patterns, fp8
(e4m3) cache bytes as ``numpy.uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# no -ffast-math, no FMA contraction: results must not depend on the host ISA
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (host ISA, no GPU)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.ora_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.ora_bf16_to_f64.restype = dbl
        lib.ora_f64_to_bf16.argtypes = [dbl]
        lib.ora_f64_to_bf16.restype = ctypes.c_uint16
        lib.ora_f64_to_bf16_array.argtypes = [P, i64, P]
        lib.ora_f64_to_bf16_array.restype = None
        lib.ora_rope.argtypes = [P, i64, i32, i32, P, P, P, i32, P, P]
        lib.ora_rope.restype = i32
        lib.ora_kv_store.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, P, i64]
        lib.ora_kv_store.restype = i32
        lib.ora_decode.argtypes = [P, i32, i32, P, P, i32, i64, i32, i32, i32,
                                   P, i32, i32, P, P, dbl, P, P, i64, P]
        lib.ora_decode.restype = i32
        lib.ora_prefill.argtypes = [P, i64, i32, P, P, i32, i64, i32, i32, i32,
                                    P, P, i32, P, i32, i32, P, dbl, P, P, i64, P]
        lib.ora_prefill.restype = i32
        lib.ora_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.ora_e4m3_to_f64.restype = dbl
        lib.ora_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.ora_f32_to_e4m3.restype = ctypes.c_uint8
        lib.ora_f32_to_e4m3_array.argtypes = [P, i64, P]
        lib.ora_f32_to_e4m3_array.restype = None
        lib.ora_kv_store_fp8.argtypes = [P, P, i32, i64, i32, i32, i32, P, P, P, i64, P, P]
        lib.ora_kv_store_fp8.restype = i32
        lib.ora_decode_fp8.argtypes = [P, i32, i32, P, P, i32, i64, i32, i32, i32,
                                       P, i32, i32, P, P, dbl, P, P, P, P, i64, P]
        lib.ora_decode_fp8.restype = i32
        lib.ora_prefill_fp8.argtypes = [P, i64, i32, P, P, i32, i64, i32, i32, i32,
                                        P, P, i32, P, i32, i32, P, dbl, P, P, P, P, i64, P]
        lib.ora_prefill_fp8.restype = i32
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what}: oracle status {rc}")


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (elementwise)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 bit patterns, nearest, ties to even."""
    x, xp = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().ora_f64_to_bf16_array(xp, x.size, out.ctypes.data_as(ctypes.c_void_p))
    return out


def rope(x_bits, positions, cos_tab, sin_tab):
    """Interleaved-pair rotary embedding of packed [T, H, D] bf16 vectors.

    Returns (y_bf16_bits, y_f64).  See ``ora_rope`` in oracle.c."""
    x, xp = _c(x_bits, np.uint16)
    T, H, D = x.shape
    pos, pp = _c(positions, np.int32)
    ct, cp = _c(cos_tab, np.float32)
    st, sp = _c(sin_tab, np.float32)
    assert ct.shape == st.shape and ct.shape[1] == D // 2
    yb = np.empty_like(x)
    yf = np.empty(x.shape, dtype=np.float64)
    rc = _load().ora_rope(xp, T, H, D, pp, cp, sp, ct.shape[0],
                          yb.ctypes.data_as(ctypes.c_void_p), yf.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "rope")
    return yb, yf


def kv_store(k_buf_bits, v_buf_bits, layer, k_new_bits, v_new_bits, loc):
    """Return copies of the two [n_layers, size, Hkv, D] buffers with the new
    tokens' rows written at ``loc``.  See ``ora_kv_store``."""
    kb = np.array(k_buf_bits, dtype=np.uint16, copy=True, order="C")
    vb = np.array(v_buf_bits, dtype=np.uint16, copy=True, order="C")
    n_layers, size, Hkv, D = kb.shape
    kn, knp = _c(k_new_bits, np.uint16)
    vn, vnp = _c(v_new_bits, np.uint16)
    lc, lp = _c(loc, np.int32)
    rc = _load().ora_kv_store(kb.ctypes.data_as(ctypes.c_void_p), vb.ctypes.data_as(ctypes.c_void_p),
                              n_layers, size, Hkv, D, layer, knp, vnp, lp, lc.size)
    _check(rc, "kv_store")
    return kb, vb


def decode(q_bits, k_buf_bits, v_buf_bits, layer, req_to_token, req_pool_indices,
           seq_lens, scale, sel=None):
    """Packed decode attention in float64.

    q [B, Hq, D]; buffers [n_layers, size, Hkv, D]; req_to_token [R, max_ctx].
    Returns out [B, Hq, D] (float64), or [n_sel, D] for ``sel`` = (b_idx, hq_idx)."""
    q, qp = _c(q_bits, np.uint16)
    B, Hq, D = q.shape
    kb, kp = _c(k_buf_bits, np.uint16)
    vb, vp = _c(v_buf_bits, np.uint16)
    n_layers, size, Hkv, D2 = kb.shape
    assert D2 == D and vb.shape == kb.shape
    r2t, rp = _c(req_to_token, np.int32)
    rpi, rpip = _c(req_pool_indices, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    if sel is None:
        out = np.empty((B, Hq, D), dtype=np.float64)
        sb = sh = None
        nsel = 0
    else:
        sbb, sb = _c(sel[0], np.int32)
        shh, sh = _c(sel[1], np.int32)
        nsel = sbb.size
        out = np.empty((nsel, D), dtype=np.float64)
    rc = _load().ora_decode(qp, B, Hq, kp, vp, n_layers, size, Hkv, D, layer,
                            rp, r2t.shape[0], r2t.shape[1], rpip, slp, float(scale),
                            sb, sh, nsel, out.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "decode")
    return out


def prefill(q_bits, k_buf_bits, v_buf_bits, layer, qo_indptr, kv_indptr, req_to_token,
            req_pool_indices, scale, sel=None):
    """Ragged causal prefill in float64 (causal mask aligned to each request's end).

    q [T, Hq, D]; indptrs [R+1]; returns out [T, Hq, D] or [n_sel, D] for
    ``sel`` = (t_idx, hq_idx)."""
    q, qp = _c(q_bits, np.uint16)
    T, Hq, D = q.shape
    kb, kp = _c(k_buf_bits, np.uint16)
    vb, vp = _c(v_buf_bits, np.uint16)
    n_layers, size, Hkv, D2 = kb.shape
    assert D2 == D and vb.shape == kb.shape
    qo, qop = _c(qo_indptr, np.int32)
    kv, kvp = _c(kv_indptr, np.int32)
    R = qo.size - 1
    r2t, rp = _c(req_to_token, np.int32)
    rpi, rpip = _c(req_pool_indices, np.int32)
    if sel is None:
        out = np.empty((T, Hq, D), dtype=np.float64)
        st = sh = None
        nsel = 0
    else:
        stt, st = _c(sel[0], np.int32)
        shh, sh = _c(sel[1], np.int32)
        nsel = stt.size
        out = np.empty((nsel, D), dtype=np.float64)
    rc = _load().ora_prefill(qp, T, Hq, kp, vp, n_layers, size, Hkv, D, layer, qop, kvp, R,
                             rp, r2t.shape[0], r2t.shape[1], rpip, float(scale),
                             st, sh, nsel, out.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "prefill")
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    """Exact values of e4m3 bytes (elementwise; NaN for 0x7F / 0xFF)."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return np.array([lib.ora_e4m3_to_f64(int(b)) for b in c.ravel()], dtype=np.float64).reshape(c.shape)


def f32_to_e4m3(x) -> np.ndarray:
    """Nearest e4m3 bytes to float32 values, ties to even, finite overflow
    saturating to +-448.  See ``ora_f32_to_e4m3``."""
    x, xp = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().ora_f32_to_e4m3_array(xp, x.size, out.ctypes.data_as(ctypes.c_void_p))
    return out


def kv_store_fp8(k_buf, v_buf, layer, k_new_bits, v_new_bits, loc, k_scale, v_scale):
    """Return copies of the two [n_layers, size, Hkv, D] byte buffers with the
    new tokens' rows quantised to e4m3 by the per-(layer, kv head) scales
    [n_layers, Hkv] and written at ``loc``.  See ``ora_kv_store_fp8``."""
    kb = np.array(k_buf, dtype=np.uint8, copy=True, order="C")
    vb = np.array(v_buf, dtype=np.uint8, copy=True, order="C")
    n_layers, size, Hkv, D = kb.shape
    kn, knp = _c(k_new_bits, np.uint16)
    vn, vnp = _c(v_new_bits, np.uint16)
    lc, lp = _c(loc, np.int32)
    ks, ksp = _c(k_scale, np.float32)
    vs, vsp = _c(v_scale, np.float32)
    assert ks.shape == (n_layers, Hkv) and vs.shape == (n_layers, Hkv)
    rc = _load().ora_kv_store_fp8(kb.ctypes.data_as(ctypes.c_void_p), vb.ctypes.data_as(ctypes.c_void_p),
                                  n_layers, size, Hkv, D, layer, knp, vnp, lp, lc.size, ksp, vsp)
    _check(rc, "kv_store_fp8")
    return kb, vb


def decode_fp8(q_bits, k_buf, v_buf, layer, req_to_token, req_pool_indices, seq_lens, scale,
               k_scale, v_scale, sel=None):
    """Packed decode attention in float64 over an e4m3 cache with per-(layer,
    kv head) scales.  Same shapes and ``sel`` as ``decode``."""
    q, qp = _c(q_bits, np.uint16)
    B, Hq, D = q.shape
    kb, kp = _c(k_buf, np.uint8)
    vb, vp = _c(v_buf, np.uint8)
    n_layers, size, Hkv, D2 = kb.shape
    assert D2 == D and vb.shape == kb.shape
    ks, ksp = _c(k_scale, np.float32)
    vs, vsp = _c(v_scale, np.float32)
    assert ks.shape == (n_layers, Hkv) and vs.shape == (n_layers, Hkv)
    r2t, rp = _c(req_to_token, np.int32)
    rpi, rpip = _c(req_pool_indices, np.int32)
    sl, slp = _c(seq_lens, np.int32)
    if sel is None:
        out = np.empty((B, Hq, D), dtype=np.float64)
        sb = sh = None
        nsel = 0
    else:
        sbb, sb = _c(sel[0], np.int32)
        shh, sh = _c(sel[1], np.int32)
        nsel = sbb.size
        out = np.empty((nsel, D), dtype=np.float64)
    rc = _load().ora_decode_fp8(qp, B, Hq, kp, vp, n_layers, size, Hkv, D, layer,
                                rp, r2t.shape[0], r2t.shape[1], rpip, slp, float(scale), ksp, vsp,
                                sb, sh, nsel, out.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "decode_fp8")
    return out


def prefill_fp8(q_bits, k_buf, v_buf, layer, qo_indptr, kv_indptr, req_to_token, req_pool_indices, scale,
                k_scale, v_scale, sel=None):
    """Ragged causal prefill in float64 over an e4m3 cache with per-(layer, kv
    head) scales.  Same shapes and ``sel`` as ``prefill``; see
    ``ora_prefill_fp8``."""
    q, qp = _c(q_bits, np.uint16)
    T, Hq, D = q.shape
    kb, kp = _c(k_buf, np.uint8)
    vb, vp = _c(v_buf, np.uint8)
    n_layers, size, Hkv, D2 = kb.shape
    assert D2 == D and vb.shape == kb.shape
    ks, ksp = _c(k_scale, np.float32)
    vs, vsp = _c(v_scale, np.float32)
    assert ks.shape == (n_layers, Hkv) and vs.shape == (n_layers, Hkv)
    qo, qop = _c(qo_indptr, np.int32)
    kv, kvp = _c(kv_indptr, np.int32)
    R = qo.size - 1
    r2t, rp = _c(req_to_token, np.int32)
    rpi, rpip = _c(req_pool_indices, np.int32)
    if sel is None:
        out = np.empty((T, Hq, D), dtype=np.float64)
        st = sh = None
        nsel = 0
    else:
        stt, st = _c(sel[0], np.int32)
        shh, sh = _c(sel[1], np.int32)
        nsel = stt.size
        out = np.empty((nsel, D), dtype=np.float64)
    rc = _load().ora_prefill_fp8(qp, T, Hq, kp, vp, n_layers, size, Hkv, D, layer, qop, kvp, R,
                                 rp, r2t.shape[0], r2t.shape[1], rpip, float(scale), ksp, vsp,
                                 st, sh, nsel, out.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "prefill_fp8")
    return out
