"""GPU parity of the tcgen05 ragged paged prefill against the float64 oracle.

Tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref| (bf16 operands, fp32 accumulation in
tensor memory, P rounded to bf16)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W
from _helpers import assert_attention_close, bits, npy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


def _run(pb, ws=None, out=None):
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes()) if ws is None else ws
    out = torch.full_like(pb.q, float("nan")) if out is None else out
    api.pa_paged_prefill_attn(pb.q, pb.kv.k_buf, pb.kv.v_buf, pb.layer, pb.qo_indptr, pb.kv_indptr,
                              pb.kv.req_to_token, pb.kv.req_pool_indices, pb.scale, ws, out)
    torch.cuda.synchronize()
    return out, ws


def _store(pb):
    """Store the raw new K/V with the library; the same on the host for the oracle."""
    kb0, vb0 = bits(pb.kv.k_buf), bits(pb.kv.v_buf)
    api.pa_kv_store(pb.kv.k_buf, pb.kv.v_buf, pb.layer, pb.k_new, pb.v_new, pb.loc)
    return oracle.kv_store(kb0, vb0, pb.layer, bits(pb.k_new), bits(pb.v_new), npy(pb.loc))


def _ref(pb, kb, vb, sel=None):
    return oracle.prefill(bits(pb.q), kb, vb, pb.layer, npy(pb.qo_indptr), npy(pb.kv_indptr),
                          npy(pb.kv.req_to_token), npy(pb.kv.req_pool_indices), pb.scale, sel=sel)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("page", [16, 1])
def test_ragged_small(G, page):
    new = [1, 31, 32, 33, 130, 7]
    pre = [0, 5, 128, 0, 300, 17]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=2 * G, n_kv_heads=2, head_dim=128,
                              size=4096, page_size=page, seed=G * 10 + page, req_rows=9, device="cuda")
    kb, vb = _store(pb)
    out, ws = _run(pb)
    assert_attention_close(npy(out.float()), _ref(pb, kb, vb), f"prefill G={G} page={page}")
    assert api.pa_get_error(ws) == 0


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("page", [16, 1])
def test_ragged_small_head_dim_64(G, page):
    new = [1, 31, 32, 33, 130, 7, 300]
    pre = [0, 5, 128, 0, 300, 17, 1000]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=2 * G, n_kv_heads=2, head_dim=64,
                              size=4096, page_size=page, seed=G * 10 + page + 64, req_rows=9, device="cuda")
    kb, vb = _store(pb)
    out, ws = _run(pb)
    assert_attention_close(npy(out.float()), _ref(pb, kb, vb), f"prefill D=64 G={G} page={page}")
    assert api.pa_get_error(ws) == 0


@pytest.mark.parametrize("G", [1, 4, 16])
def test_dense_prefill_head_dim_64(G):
    new = [1, 17, 300, 128, 700]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=[0] * len(new), n_q_heads=2 * G, n_kv_heads=2,
                              head_dim=64, size=4096, page_size=16, seed=70 + G, device="cuda")
    kb, vb = _store(pb)
    ref, _ = _run(pb)
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    out = torch.full_like(pb.q, float("nan"))
    api.pa_dense_prefill_attn(pb.q, pb.k_new, pb.v_new, pb.qo_indptr, pb.scale, ws, out)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert_attention_close(npy(out.float()), _ref(pb, kb, vb), f"dense prefill D=64 G={G}")


def test_mixed_pages_and_long_prefix():
    # page size 4: 16-position groups are never one contiguous page -> per-row boxes
    new, pre = [200, 64, 1000], [1024, 0, 40]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=32, n_kv_heads=8, head_dim=128,
                              size=16384, page_size=4, seed=7, device="cuda")
    kb, vb = _store(pb)
    out, ws = _run(pb)
    assert_attention_close(npy(out.float()), _ref(pb, kb, vb), "page 4")
    assert api.pa_get_error(ws) == 0


def test_deterministic_graph_replay_and_padding_rows_untouched():
    new, pre = [77, 300], [10, 500]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=32, n_kv_heads=8, head_dim=128,
                              size=8192, page_size=16, seed=9, device="cuda")
    kb, vb = _store(pb)
    out1, ws = _run(pb)
    out2, _ = _run(pb, ws=ws)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    og = torch.zeros_like(pb.q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.pa_paged_prefill_attn(pb.q, pb.kv.k_buf, pb.kv.v_buf, 0, pb.qo_indptr, pb.kv_indptr,
                                  pb.kv.req_to_token, pb.kv.req_pool_indices, pb.scale, ws, og, stream=s)
    for _ in range(3):
        og.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), og.view(torch.int16))
    # the work queue in the workspace header is back at zero after every launch
    words = ws.view(torch.int32)
    assert int(words[16]) == 0 and int(words[32]) == 0
    # a pack of one request writes only its own rows
    T = pb.q.shape[0]
    out = torch.full_like(pb.q, 7.0)
    one_qo = torch.tensor([0, 77], dtype=torch.int32, device="cuda")
    one_kv = torch.tensor([0, 87], dtype=torch.int32, device="cuda")
    api.pa_paged_prefill_attn(pb.q, pb.kv.k_buf, pb.kv.v_buf, 0, one_qo, one_kv, pb.kv.req_to_token,
                              pb.kv.req_pool_indices[:1].contiguous(), pb.scale, ws, out)
    torch.cuda.synchronize()
    assert torch.equal(out[:77].view(torch.int16), out1[:77].view(torch.int16))
    assert (out[77:T] == 7.0).all()
    assert int(words[16]) == 0 and int(words[32]) == 0


def test_invalid_request_is_skipped_and_flagged():
    new, pre = [20, 20], [5, 5]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=8, n_kv_heads=2, head_dim=128,
                              size=1024, page_size=16, seed=11, device="cuda")
    kb, vb = _store(pb)
    bad_kv = torch.tensor([0, 25, 35], dtype=torch.int32, device="cuda")   # request 1: L=10 < n=20
    out = torch.full_like(pb.q, 3.0)
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    api.pa_paged_prefill_attn(pb.q, pb.kv.k_buf, pb.kv.v_buf, 0, pb.qo_indptr, bad_kv, pb.kv.req_to_token,
                              pb.kv.req_pool_indices, pb.scale, ws, out)
    assert api.pa_get_error(ws) & api.DEVERR_LEN
    ref = _ref(pb, kb, vb)
    assert_attention_close(npy(out.float())[:20], ref[:20], "valid request")
    assert (out[20:] == 3.0).all()


def test_config4_full_size_sampled():
    """16 packed prompts: RoPE -> KV store -> prefill through the library; the
    oracle checks every head of 6 rows per request (first, last, 4 random)."""
    pb = W.config4(device="cuda")
    kb0, vb0 = bits(pb.kv.k_buf), bits(pb.kv.v_buf)
    q, k_new = pb.q.clone(), pb.k_new.clone()
    api.pa_rope_packed(q, k_new, pb.positions, pb.cos_tab, pb.sin_tab)
    api.pa_kv_store(pb.kv.k_buf, pb.kv.v_buf, 0, k_new, pb.v_new, pb.loc)
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    out = torch.full_like(q, float("nan"))
    api.pa_paged_prefill_attn(q, pb.kv.k_buf, pb.kv.v_buf, 0, pb.qo_indptr, pb.kv_indptr, pb.kv.req_to_token,
                              pb.kv.req_pool_indices, pb.scale, ws, out)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    assert torch.isfinite(out.float()).all()
    pos, ct, sn = npy(pb.positions), npy(pb.cos_tab), npy(pb.sin_tab)
    qr, _ = oracle.rope(bits(pb.q), pos, ct, sn)
    kr, _ = oracle.rope(bits(pb.k_new), pos, ct, sn)
    kb, vb = oracle.kv_store(kb0, vb0, 0, kr, bits(pb.v_new), npy(pb.loc))
    qo = npy(pb.qo_indptr)
    rng = np.random.default_rng(4)
    rows = []
    for r in range(len(pb.new_lens)):
        rows += [qo[r], qo[r + 1] - 1] + rng.integers(qo[r], qo[r + 1], 4).tolist()
    rows = sorted(set(int(x) for x in rows))
    Hq = q.shape[1]
    st = np.repeat(np.array(rows, np.int32), Hq)
    sh = np.tile(np.arange(Hq, dtype=np.int32), len(rows))
    ref = oracle.prefill(qr, kb, vb, 0, qo, npy(pb.kv_indptr), npy(pb.kv.req_to_token),
                         npy(pb.kv.req_pool_indices), pb.scale, sel=(st, sh))
    got = npy(out.float())[st, sh]
    assert_attention_close(got, ref, "config 4 sampled")


def test_last_rows_gathered_by_the_epilogue():
    new, pre = [1, 31, 200, 64, 129], [0, 40, 300, 0, 17]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=32, n_kv_heads=8, head_dim=128, size=8192,
                              page_size=16, seed=21, device="cuda")
    kb, vb = _store(pb)
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    R = len(new)
    out = torch.full_like(pb.q, float("nan"))
    last = torch.full((R,) + tuple(pb.q.shape[1:]), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.pa_paged_prefill_attn(pb.q, pb.kv.k_buf, pb.kv.v_buf, 0, pb.qo_indptr, pb.kv_indptr, pb.kv.req_to_token,
                              pb.kv.req_pool_indices, pb.scale, ws, out, last_out=last)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    # each request's last row against the oracle, every head, from the
    # host-built cache
    Hq = pb.q.shape[1]
    last_rows = npy(pb.qo_indptr)[1:] - 1
    sel = (np.repeat(last_rows.astype(np.int32), Hq), np.tile(np.arange(Hq, dtype=np.int32), R))
    ref_last = _ref(pb, kb, vb, sel=sel).reshape(R, Hq, -1)
    assert_attention_close(npy(last.float()), ref_last, "last rows gathered by the epilogue")
    # the gather is a copy of those rows of out, and changes nothing else
    plain, _ = _run(pb)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))
    rows = (pb.qo_indptr[1:] - 1).long()
    assert torch.equal(last.view(torch.int16), out[rows].view(torch.int16))


@pytest.mark.parametrize("G", [1, 4, 16])
def test_dense_prefill_equals_paged_prefill_without_prefix(G):
    new = [1, 17, 300, 128, 1000, 65]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=[0] * len(new), n_q_heads=2 * G, n_kv_heads=2,
                              head_dim=128, size=4096, page_size=16, seed=30 + G, device="cuda")
    kb, vb = _store(pb)
    ref, _ = _run(pb)
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    out = torch.full_like(pb.q, float("nan"))
    last = torch.full((len(new),) + tuple(pb.q.shape[1:]), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.pa_dense_prefill_attn(pb.q, pb.k_new, pb.v_new, pb.qo_indptr, pb.scale, ws, out, last_out=last)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(last.view(torch.int16), ref[(pb.qo_indptr[1:] - 1).long()].view(torch.int16))
    assert_attention_close(npy(out.float()), _ref(pb, kb, vb), f"dense prefill G={G}")
