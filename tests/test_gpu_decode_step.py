"""The fused decode step (RoPE + KV store + decode attention in one launch)
against the three separate calls and against the float64 oracle.

pa_decode_step must give the same bits as pa_rope_packed -> pa_kv_store ->
pa_paged_decode_attn: the same rotated q (in registers), the same rotated K
and V rows in the cache, the same attention plan.  The oracle check is the
usual tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W
from _helpers import assert_attention_close, bits, npy

pytestmark = pytest.mark.gpu
MAX_SPLITS = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


def _state(lens, hq, hkv, d, page, seed, size=16384):
    return W.make_decode_step(lens=lens, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, n_layers=2, size=size,
                              page_size=page, seed=seed, layer=1, max_ctx=max(lens) + 16, device="cuda")


def _chain(st, ws, out):
    q, k = st.q.clone(), st.k_new.clone()
    api.pa_rope_packed(q, k, st.positions, st.cos_tab, st.sin_tab)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, k, st.v_new, st.loc)
    api.pa_paged_decode_attn(q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token, st.kv.req_pool_indices,
                             st.kv.seq_lens, st.scale, ws, MAX_SPLITS, out)


def _step(st, ws, out, loc=None):
    api.pa_decode_step(st.q, st.k_new, st.v_new, st.positions, st.cos_tab, st.sin_tab, st.kv.k_buf, st.kv.v_buf,
                       st.layer, st.loc if loc is None else loc, st.kv.req_to_token, st.kv.req_pool_indices,
                       st.kv.seq_lens, st.scale, ws, MAX_SPLITS, out)


@pytest.mark.parametrize("hq,hkv,d,page", [(32, 8, 128, 16), (32, 8, 128, 1), (64, 8, 128, 16), (16, 1, 128, 16),
                                           (8, 2, 64, 16), (8, 2, 64, 1)])
def test_fused_step_bit_identical_to_three_calls(hq, hkv, d, page):
    lens = [3000, 17, 1, 1200, 640, 16, 4097]
    st = _state(lens, hq, hkv, d, page, seed=hq + hkv + d + page)
    B = len(lens)
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, hq, hkv, d, MAX_SPLITS))
    kb0, vb0 = st.kv.k_buf.clone(), st.kv.v_buf.clone()
    q0, k0 = st.q.clone(), st.k_new.clone()
    ref = torch.full_like(st.q, float("nan"))
    _chain(st, ws, ref)
    torch.cuda.synchronize()
    kb_ref, vb_ref = st.kv.k_buf.clone(), st.kv.v_buf.clone()
    st.kv.k_buf.copy_(kb0)
    st.kv.v_buf.copy_(vb0)
    got = torch.full_like(st.q, float("nan"))
    _step(st, ws, got)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(st.kv.k_buf.view(torch.int16), kb_ref.view(torch.int16))     # whole buffers, canaries too
    assert torch.equal(st.kv.v_buf.view(torch.int16), vb_ref.view(torch.int16))
    assert torch.equal(st.q, q0) and torch.equal(st.k_new, k0)                      # inputs only read


def test_fused_step_largest_batch_bit_identical_to_three_calls():
    # 4096 requests x 16 kv heads, one split each: 65536 items, more than 256
    # per CTA, so items past a CTA's first 256 read their position from global
    # memory; every item's new rows go through its own tile
    B, hq, hkv, d = 4096, 16, 16, 64
    rng = np.random.default_rng(8)
    lens = [int(x) for x in rng.integers(1, 41, size=B)]
    st = _state(lens, hq, hkv, d, 16, seed=8, size=B * 48)
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, hq, hkv, d, MAX_SPLITS))
    kb0, vb0 = st.kv.k_buf.clone(), st.kv.v_buf.clone()
    ref = torch.full_like(st.q, float("nan"))
    _chain(st, ws, ref)
    torch.cuda.synchronize()
    kb_ref, vb_ref = st.kv.k_buf.clone(), st.kv.v_buf.clone()
    st.kv.k_buf.copy_(kb0)
    st.kv.v_buf.copy_(vb0)
    got = torch.full_like(st.q, float("nan"))
    _step(st, ws, got)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(st.kv.k_buf.view(torch.int16), kb_ref.view(torch.int16))
    assert torch.equal(st.kv.v_buf.view(torch.int16), vb_ref.view(torch.int16))


def test_fused_step_against_oracle_and_graph_replay():
    lens = [2500, 33, 900, 1]
    st = _state(lens, 32, 8, 128, 16, seed=77)
    B = len(lens)
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    pos, ct, sn = npy(st.positions), npy(st.cos_tab), npy(st.sin_tab)
    qr, _ = oracle.rope(bits(st.q), pos, ct, sn)
    kr, _ = oracle.rope(bits(st.k_new), pos, ct, sn)
    kb, vb = oracle.kv_store(kb0, vb0, st.layer, kr, bits(st.v_new), npy(st.loc))
    ref = oracle.decode(qr, kb, vb, st.layer, npy(st.kv.req_to_token), npy(st.kv.req_pool_indices),
                        npy(st.kv.seq_lens), st.scale)
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, 32, 8, 128, MAX_SPLITS))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    out = torch.zeros_like(st.q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.pa_decode_step(st.q, st.k_new, st.v_new, st.positions, st.cos_tab, st.sin_tab, st.kv.k_buf,
                           st.kv.v_buf, st.layer, st.loc, st.kv.req_to_token, st.kv.req_pool_indices,
                           st.kv.seq_lens, st.scale, ws, MAX_SPLITS, out, stream=s)
    first = None
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        if first is None:
            first = out.clone()
            assert_attention_close(npy(out.float()), ref, "fused decode step vs oracle")
            assert np.array_equal(bits(st.kv.k_buf), kb) and np.array_equal(bits(st.kv.v_buf), vb)
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert api.pa_get_error(ws) == 0


def test_fused_step_flags_a_loc_that_is_not_the_last_position():
    lens = [300, 200]
    st = _state(lens, 32, 8, 128, 16, seed=5)
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(2, 32, 8, 128, MAX_SPLITS))
    used = set(st.kv.used_slots.cpu().tolist())
    free = next(x for x in range(16384) if x not in used)
    bad = st.loc.clone()
    bad[1] = free                              # an unused slot, not request 1's last position
    out = torch.empty_like(st.q)
    _step(st, ws, out, loc=bad)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) & api.DEVERR_SLOT
