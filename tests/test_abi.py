"""CPU checks of the C ABI: the library loads, exports every symbol the header
declares, sizes workspaces consistently, and rejects bad arguments on the host
before any launch (these calls return before touching the CUDA runtime)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return api.lib()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "pagedattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert "pa_paged_decode_attn" in syms and "pa_paged_prefill_attn" in syms
    for s in syms:
        assert hasattr(lib, s), s
    assert set(api.EXPORTS) == set(syms)


def test_status_strings(lib):
    for code in range(8):
        assert lib.pa_status_string(code).decode().startswith(api.STATUS[code])


def test_decode_workspace_size_monotone_and_sufficient(lib):
    small = api.pa_decode_workspace_bytes(1, 32, 8, 128, 64)
    big = api.pa_decode_workspace_bytes(256, 64, 8, 128, 64)
    assert 0 < small < big
    # o_part + ml_part + counters for 256 requests at least
    assert big >= 256 * 64 * 64 * 128 * 4
    assert api.pa_decode_workspace_bytes(0, 32, 8, 128, 0) == 0
    assert api.pa_prefill_workspace_bytes() >= 256


FAKE = 0x10000000  # a 256-byte aligned non-null address; the calls below fail before using it


def _shape(n_layers=2, size=64, hkv=2, d=64):
    return api.KvShape(n_layers, size, hkv, d)


def _decode(lib, **kw):
    a = dict(q=FAKE, batch=1, hq=8, k=FAKE, v=FAKE, s=_shape(), layer=0, r2t=FAKE, rows=1, max_ctx=16,
             rpi=FAKE, sl=FAKE, scale=0.125, ws=FAKE, ws_bytes=api.pa_decode_workspace_bytes(1, 8, 2, 64, 4),
             splits=4, out=FAKE)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.pa_paged_decode_attn(P(a["q"]), a["batch"], a["hq"], P(a["k"]), P(a["v"]), a["s"], a["layer"],
                                    P(a["r2t"]), a["rows"], a["max_ctx"], P(a["rpi"]), P(a["sl"]), a["scale"],
                                    P(a["ws"]), a["ws_bytes"], a["splits"], P(a["out"]), None)


def test_decode_host_validation(lib):
    assert _decode(lib, layer=2) == 2                        # layer out of range
    assert _decode(lib, hq=7) == 2                           # Hq not a multiple of Hkv
    assert _decode(lib, s=_shape(d=96)) == 4                 # unsupported head_dim
    assert _decode(lib, hq=64) == 4                          # G = 32 > 16
    assert _decode(lib, splits=0) == 2
    assert _decode(lib, splits=129) == 2
    assert _decode(lib, batch=4097) == 2
    assert _decode(lib, ws=0) == 1
    assert _decode(lib, ws=FAKE + 16) == 3                   # workspace must be 256-byte aligned
    assert _decode(lib, ws_bytes=100) == 5
    assert _decode(lib, batch=2) == 5                        # workspace sized for one request
    assert _decode(lib, q=0) == 1
    assert _decode(lib, q=FAKE + 2) == 3
    assert _decode(lib, out=FAKE + 8) == 3
    assert _decode(lib, sl=FAKE + 1) == 3
    assert _decode(lib, batch=0, q=0, out=0) == 0            # empty batch: nothing to do


def test_store_and_rope_host_validation(lib):
    P = ctypes.c_void_p
    assert lib.pa_kv_store(P(FAKE), P(FAKE), _shape(), 2, P(FAKE), P(FAKE), P(FAKE), 4, None, None) == 2
    assert lib.pa_kv_store(P(FAKE), P(FAKE), _shape(d=12), 0, P(FAKE), P(FAKE), P(FAKE), 4, None, None) == 4
    assert lib.pa_kv_store(P(FAKE), None, _shape(), 0, P(FAKE), P(FAKE), P(FAKE), 4, None, None) == 1
    assert lib.pa_kv_store(P(FAKE + 4), P(FAKE), _shape(), 0, P(FAKE), P(FAKE), P(FAKE), 4, None, None) == 3
    assert lib.pa_kv_store(None, None, _shape(), 0, None, None, None, 0, None, None) == 0
    assert lib.pa_rope_packed(P(FAKE), 4, P(FAKE), 2, 10, P(FAKE), 3, P(FAKE), P(FAKE), 16, None, None) == 4
    assert lib.pa_rope_packed(P(FAKE), 4, None, 2, 64, P(FAKE), 3, P(FAKE), P(FAKE), 16, None, None) == 1
    assert lib.pa_rope_packed(P(FAKE), 4, P(FAKE), 2, 64, P(FAKE), 3, P(FAKE + 4), P(FAKE), 16, None, None) == 3
    assert lib.pa_rope_packed(P(FAKE), 4, P(FAKE), 2, 64, P(FAKE), -1, P(FAKE), P(FAKE), 16, None, None) == 2
    assert lib.pa_workspace_init(None, 1024, None) == 1
    assert lib.pa_workspace_init(P(FAKE + 8), 1024, None) == 3


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        api.lib()


def test_launch_overlap_mode_switch(lib):
    assert api.pa_get_launch_overlap() == api.OVERLAP_OFF
    try:
        for m in (api.OVERLAP_SAFE, api.OVERLAP_EARLY_METADATA, api.OVERLAP_EARLY_KV, api.OVERLAP_OFF):
            api.pa_set_launch_overlap(m)
            assert api.pa_get_launch_overlap() == m
        assert lib.pa_set_launch_overlap(4) == 2
        assert lib.pa_set_launch_overlap(-1) == 2
        assert api.pa_get_launch_overlap() == api.OVERLAP_OFF   # a rejected mode changes nothing
    finally:
        api.pa_set_launch_overlap(api.OVERLAP_OFF)


def test_decode_step_host_validation(lib):
    P = ctypes.c_void_p
    ws_bytes = api.pa_decode_workspace_bytes(1, 8, 2, 64, 4)

    def call(**kw):
        a = dict(q=FAKE, kn=FAKE, vn=FAKE, pos=FAKE, cos=FAKE, sin=FAKE, max_pos=64, loc=FAKE, ws=FAKE)
        a.update(kw)
        return lib.pa_decode_step(P(a["q"]), P(a["kn"]), P(a["vn"]), 1, 8, P(a["pos"]), P(a["cos"]), P(a["sin"]),
                                  a["max_pos"], P(FAKE), P(FAKE), _shape(), 0, P(a["loc"]), P(FAKE), 1, 16, P(FAKE),
                                  P(FAKE), 0.125, P(a["ws"]), ws_bytes, 4, P(FAKE), None)
    assert call(kn=0) == 1
    assert call(loc=0) == 1
    assert call(cos=0) == 1
    assert call(max_pos=0) == 2
    assert call(vn=FAKE + 8) == 3                 # k_new / v_new must be 16-byte aligned
    assert call(pos=FAKE + 2) == 3
    assert call(ws=FAKE + 16) == 3


def test_prefill_variants_host_validation(lib):
    P = ctypes.c_void_p
    ws_bytes = api.pa_prefill_workspace_bytes()
    rc = lib.pa_paged_prefill_attn_last(P(FAKE), 10, 8, P(FAKE), P(FAKE), api.KvShape(1, 64, 2, 128), 0, P(FAKE),
                                        P(FAKE), 1, P(FAKE), 1, 16, P(FAKE), 0.1, P(FAKE), ws_bytes, P(FAKE), None, None)
    assert rc == 1                                              # last_out is required
    dense = lambda **kw: lib.pa_dense_prefill_attn(P(FAKE), 10, kw.get("hq", 8), P(FAKE), P(FAKE), kw.get("hkv", 2),
                                                   kw.get("d", 128), P(FAKE), 1, 0.1, P(kw.get("ws", FAKE)), ws_bytes,
                                                   P(FAKE), P(kw.get("last", 0)), None)
    assert dense(d=96) == 4
    assert dense(d=32) == 4
    assert dense(hq=6, hkv=4) == 2
    assert dense(ws=0) == 1
    assert dense(last=FAKE + 8) == 3


def test_cascade_workspace_and_validation(lib):
    caps = (32, 4, 8, 64)
    small = api.pa_cascade_workspace_bytes(*caps, 32, 8, 128)
    assert small >= api.pa_decode_workspace_bytes(32, 32, 8, 128, 64)
    assert api.pa_cascade_workspace_bytes(64, 8, 8, 64, 32, 8, 128) > small
    assert api.pa_cascade_workspace_bytes(32, 4, 0, 64, 32, 8, 128) == 0        # max_group_size >= 1
    assert api.pa_cascade_workspace_bytes(32, 4096, 64, 64, 32, 8, 128) == 0    # virtual batch over 4096
    P = ctypes.c_void_p
    c = api.CascadeCaps(*caps)
    call = lambda **kw: lib.pa_paged_decode_attn_cascade(
        P(FAKE), kw.get("b", 1), 32, P(FAKE), P(FAKE), api.KvShape(1, 64, 8, 128), 0, P(FAKE), 1, 16, P(FAKE),
        P(FAKE), P(kw.get("ip", FAKE)), P(FAKE), P(FAKE), kw.get("ng", 1), c, 0.1, P(FAKE), kw.get("wsb", small),
        P(FAKE), None)
    assert call(b=33) == 2                        # batch over caps.max_batch
    assert call(ng=5) == 2                        # groups over caps.max_groups
    assert call(wsb=small - 1) == 5
    assert call(ip=0) == 1
    assert call(ip=FAKE + 2) == 3


def test_fp8_entry_points_host_validation(lib):
    P = ctypes.c_void_p

    def store(s=None, layer=0, ks=FAKE, vs=FAKE, n=4, k=FAKE):
        return lib.pa_kv_store_fp8(P(k), P(FAKE), s or _shape(d=64), layer, P(FAKE), P(FAKE), P(FAKE), n,
                                   P(ks) if ks else None, P(vs) if vs else None, None, None)

    assert store(layer=2) == 2
    assert store(s=_shape(d=8)) == 4                         # head_dim must be a multiple of 16
    assert store(ks=0) == 1
    assert store(vs=FAKE + 2) == 3
    assert store(k=FAKE + 8) == 3                            # 16-byte aligned buffers
    assert store(n=0, ks=0, vs=0) == 0                       # no tokens: nothing to do

    def dec(batch=1, ks=FAKE, vs=FAKE, s=None, hq=8):
        return lib.pa_paged_decode_attn_fp8(
            P(FAKE), batch, hq, P(FAKE), P(FAKE), s or _shape(), 0, P(FAKE), 1, 16, P(FAKE), P(FAKE), 0.125,
            P(ks) if ks else None, P(vs) if vs else None, P(FAKE), api.pa_decode_workspace_bytes(1, 8, 2, 64, 4),
            4, P(FAKE), None)

    assert dec(ks=0) == 1
    assert dec(vs=FAKE + 1) == 3
    assert dec(s=_shape(d=96)) == 4
    assert dec(hq=7) == 2
    assert dec(batch=2) == 5                                 # workspace sized for one request
    assert dec(batch=0, ks=0, vs=0) == 0


def test_fp8_wrappers_reject_wrong_cache_dtypes_before_the_library():
    import torch
    bf = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16)
    sc = torch.ones((1, 1), dtype=torch.float32)
    with pytest.raises(TypeError, match="uint8 or float8_e4m3fn"):
        api.pa_kv_store_fp8(bf, bf, 0, None, None, None, sc, sc)
    with pytest.raises(TypeError, match="uint8 or float8_e4m3fn"):
        api.pa_paged_decode_attn_fp8(None, bf, bf, 0, None, None, None, 0.1, sc, sc, None, 4, None)
    u8 = torch.zeros((1, 4, 1, 64), dtype=torch.uint8)
    with pytest.raises(TypeError, match="CUDA tensor"):            # host memory is never passed down
        api.pa_kv_store_fp8(u8, u8, 0, None, None, None, sc, sc)


def test_noalloc_validation_runs_before_any_cuda_call(lib):
    # On a machine without a GPU, a call that got past validation would fail
    # in the CUDA runtime (PA_ERR_CUDA); each of these must instead return its
    # validation error, so nothing was enqueued or written.
    P = ctypes.c_void_p

    def call(**kw):
        a = dict(q=FAKE, batch=1, hq=8, s=_shape(), layer=0, splits=4, out=FAKE, err=None)
        a.update(kw)
        return lib.pa_paged_decode_attn_noalloc(P(a["q"]), a["batch"], a["hq"], P(FAKE), P(FAKE), a["s"], a["layer"],
                                                P(FAKE), 1, 16, P(FAKE), P(FAKE), 0.125, a["splits"], P(a["out"]),
                                                P(a["err"]) if a["err"] else None, None)
    assert call(q=0) == 1                         # null q
    assert call(out=FAKE + 8) == 3
    assert call(s=_shape(d=96)) == 4              # unsupported head_dim
    assert call(hq=64) == 4                       # G = 32 > 16
    assert call(hq=7) == 2
    assert call(layer=2) == 2
    assert call(splits=129) == 2
    assert call(batch=4000, hq=32, s=_shape(hkv=8, d=128), splits=64) == 5   # beyond the 16 MiB array
    assert call(err=FAKE + 2) == 3
    assert call(batch=0, q=0, out=0) == 0


def test_wait_timeout_hook_round_trip(lib):
    assert api.pa_get_wait_timeout_ns() == api.WAIT_TIMEOUT_DEFAULT_NS
    try:
        api.pa_set_wait_timeout_ns(0)
        assert api.pa_get_wait_timeout_ns() == 0
        api.pa_set_wait_timeout_ns(12345)
        assert api.pa_get_wait_timeout_ns() == 12345
    finally:
        api.pa_set_wait_timeout_ns(api.WAIT_TIMEOUT_DEFAULT_NS)
    assert api.pa_get_wait_timeout_ns() == api.WAIT_TIMEOUT_DEFAULT_NS


def test_prefill_fp8_host_validation(lib):
    P = ctypes.c_void_p
    ws_bytes = api.pa_prefill_workspace_bytes()

    def call(d=128, hq=8, ks=FAKE, vs=FAKE, n=10, ws=FAKE):
        return lib.pa_paged_prefill_attn_fp8(P(FAKE), n, hq, P(FAKE), P(FAKE), api.KvShape(1, 64, 2, d), 0, P(FAKE),
                                             P(FAKE), 1, P(FAKE), 1, 16, P(FAKE), 0.1, P(ks) if ks else None,
                                             P(vs) if vs else None, P(ws), ws_bytes, P(FAKE), None)
    assert call(d=96) == 4
    assert call(hq=7) == 2
    assert call(hq=6) == 4                        # G = 3
    assert call(ks=0) == 1
    assert call(vs=FAKE + 2) == 3
    assert call(ws=FAKE + 16) == 3
    assert call(n=0, ks=0, vs=0) == 0
