"""GPU parity of packed split-KV decode attention against the float64 oracle.

All calls go through the C ABI (ctypes binding).  Tolerance: |gpu - ref| <=
1e-2 + 1e-2 |ref| elementwise (bf16 inputs, fp32 accumulation, bf16 output).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W
from _helpers import assert_attention_close, bits, compact_requests, npy

pytestmark = pytest.mark.gpu
MAX_SPLITS = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


def _ws(B, Hq, Hkv, D, max_splits=MAX_SPLITS):
    return api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, Hkv, D, max_splits))


def _oracle_full(st, kb, vb, q_bits=None):
    return oracle.decode(bits(st.q) if q_bits is None else q_bits, kb, vb, st.layer, npy(st.kv.req_to_token),
                         npy(st.kv.req_pool_indices), npy(st.kv.seq_lens), st.scale)


def _store_raw(st):
    """Store the step's raw new K/V (no rotary) with the library call, and the same on the host."""
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    return oracle.kv_store(kb0, vb0, st.layer, bits(st.k_new), bits(st.v_new), npy(st.loc))


def _decode(st, max_splits=MAX_SPLITS, ws=None):
    B, Hq, D = st.q.shape
    ws = _ws(B, Hq, st.kv.k_buf.shape[2], D, max_splits) if ws is None else ws
    out = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                             st.kv.req_pool_indices, st.kv.seq_lens, st.scale, ws, max_splits, out)
    torch.cuda.synchronize()
    return out, ws


def test_config1_full_step():
    """Config 1 end to end: RoPE -> KV store -> decode, all through the library."""
    st = W.config1(device="cuda")
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    q, k_new = st.q.clone(), st.k_new.clone()
    api.pa_rope_packed(q, k_new, st.positions, st.cos_tab, st.sin_tab)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, 0, k_new, st.v_new, st.loc)
    ws = _ws(1, 8, 2, 64)
    out = torch.empty_like(q)
    api.pa_paged_decode_attn(q, st.kv.k_buf, st.kv.v_buf, 0, st.kv.req_to_token, st.kv.req_pool_indices,
                             st.kv.seq_lens, st.scale, ws, MAX_SPLITS, out)
    torch.cuda.synchronize()
    pos, ct, sn = npy(st.positions), npy(st.cos_tab), npy(st.sin_tab)
    qr, _ = oracle.rope(bits(st.q), pos, ct, sn)
    kr, _ = oracle.rope(bits(st.k_new), pos, ct, sn)
    kb, vb = oracle.kv_store(kb0, vb0, 0, kr, bits(st.v_new), npy(st.loc))
    ref = oracle.decode(qr, kb, vb, 0, npy(st.kv.req_to_token), npy(st.kv.req_pool_indices),
                        npy(st.kv.seq_lens), st.scale)
    assert_attention_close(npy(out.float()), ref, "config 1")
    assert api.pa_get_error(ws) == 0


@pytest.mark.parametrize("Hq,Hkv,D,page", [(8, 2, 64, 16), (32, 8, 128, 16), (64, 8, 128, 1), (16, 1, 128, 4),
                                           (4, 4, 64, 1), (32, 2, 128, 16)])
def test_ragged_batch(Hq, Hkv, D, page):
    lens = [1, 15, 16, 17, 63, 64, 65, 300, 1023, 1024, 1025, 2500]
    st = W.make_decode_step(lens=lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_layers=2, size=16384,
                            page_size=page, seed=Hq * 7 + D + page, layer=1, req_rows=20, max_ctx=2600,
                            device="cuda")
    kb, vb = _store_raw(st)
    out, ws = _decode(st)
    assert_attention_close(npy(out.float()), _oracle_full(st, kb, vb), f"ragged Hq={Hq} Hkv={Hkv} D={D}")
    assert api.pa_get_error(ws) == 0


@pytest.mark.parametrize("max_splits", [1, 2, 3, 8, 64, 128])
def test_split_count_invariance(max_splits):
    """Any split cap gives the oracle's result; caps below the planned count
    stretch splits beyond the plan's longest split (2048 tokens)."""
    lens = [5000, 3, 2048, 777]
    st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=1, size=16384,
                            page_size=16, seed=123, req_rows=4, max_ctx=5000, device="cuda")
    kb, vb = _store_raw(st)
    out, _ = _decode(st, max_splits=max_splits)
    assert_attention_close(npy(out.float()), _oracle_full(st, kb, vb), f"max_splits={max_splits}")


def test_empty_and_zero_batch():
    st = W.make_decode_step(lens=[0, 7, 0], n_q_heads=8, n_kv_heads=2, head_dim=64, n_layers=1, size=256,
                            page_size=16, seed=5, device="cuda")
    # seq_len 0 requests have no token to store: store only request 1's token
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, 0, st.k_new[1:2].contiguous(), st.v_new[1:2].contiguous(),
                    st.loc[1:2].contiguous())
    kb, vb = oracle.kv_store(kb0, vb0, 0, bits(st.k_new)[1:2], bits(st.v_new)[1:2], npy(st.loc)[1:2])
    out, ws = _decode(st)
    ref = _oracle_full(st, kb, vb)
    assert not ref[0].any() and not ref[2].any()
    assert_attention_close(npy(out.float()), ref, "empty requests")
    assert (npy(out[0].float()) == 0).all() and (npy(out[2].float()) == 0).all()
    # batch 0 is a no-op
    e = torch.empty(0, 8, 64, dtype=torch.bfloat16, device="cuda")
    api.pa_paged_decode_attn(e, st.kv.k_buf, st.kv.v_buf, 0, st.kv.req_to_token, st.kv.req_pool_indices[:0],
                             st.kv.seq_lens[:0], st.scale, ws, MAX_SPLITS, e)


def test_deterministic_and_graph_replay_bit_exact():
    lens = [4000, 1500, 9, 8192]
    st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=1, size=32768,
                            page_size=16, seed=77, max_ctx=8192, device="cuda")
    _store_raw(st)
    out1, ws = _decode(st)
    out2, _ = _decode(st, ws=ws)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    out_g = torch.empty_like(st.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.pa_paged_decode_attn(st.q, st.kv.k_buf, st.kv.v_buf, 0, st.kv.req_to_token, st.kv.req_pool_indices,
                                 st.kv.seq_lens, st.scale, ws, MAX_SPLITS, out_g, stream=s)
    for _ in range(3):
        out_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), out_g.view(torch.int16))
    # new lengths in place (the graph reads them on the device): still exact vs eager
    st.kv.seq_lens.copy_(torch.tensor([3000, 1500, 9, 100], dtype=torch.int32, device="cuda"))
    g.replay()
    out3, _ = _decode(st, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(out3.view(torch.int16), out_g.view(torch.int16))


def test_batch_changes_within_one_workspace():
    ws = _ws(16, 32, 8, 128)
    for i, lens in enumerate([[3000] * 16, [50, 4000], [1] * 9, [2047, 2049, 4096]]):
        st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=1, size=65536,
                                page_size=16, seed=300 + i, device="cuda")
        kb, vb = _store_raw(st)
        out, _ = _decode(st, ws=ws)
        assert_attention_close(npy(out.float()), _oracle_full(st, kb, vb), f"refill {i}")
    assert api.pa_get_error(ws) == 0


def test_large_batch_of_tiny_requests_matches_oracle():
    # a large batch (many items per CTA, deferred merge) of tiny requests:
    # most items have fewer tiles than warps, so most warps' load cursors skip
    # many items in a row; the whole output against the oracle, twice
    B = 1024
    lens = [int(x) for x in np.random.default_rng(17).integers(1, 61, size=B)]
    st = W.make_decode_step(lens=lens, n_q_heads=16, n_kv_heads=8, head_dim=64, n_layers=1, size=B * 64,
                            page_size=16, seed=17, max_ctx=64, device="cuda")
    kb, vb = _store_raw(st)
    ref = _oracle_full(st, kb, vb)
    ws = _ws(B, 16, 8, 64)
    for _ in range(2):
        out, _ = _decode(st, ws=ws)
        assert_attention_close(npy(out.float()), ref, "tiny requests, idle warps")
    assert api.pa_get_error(ws) == 0


@pytest.mark.parametrize("case", ["mixed_d128", "mixed_d64", "one_long_hkv1", "one_long_hkv1_capped"])
def test_balanced_large_batch_plan_matches_oracle(case):
    """Large batches (2 B Hkv above the SM count) take the balanced plan: equal
    tile ranges per CTA over the (kv head, request) segments, a segment's
    pieces merged by the second kernel.  Lengths 0, 1 and tile edges, a long
    request cut into many pieces, and (capped) the fallback when a segment
    would need more pieces than max_splits; twice, bit-identical."""
    rng = np.random.default_rng({"mixed_d128": 31, "mixed_d64": 32, "one_long_hkv1": 33,
                                 "one_long_hkv1_capped": 33}[case])
    max_splits = 8 if case == "one_long_hkv1_capped" else MAX_SPLITS
    if case.startswith("mixed"):
        B, Hq, Hkv, D = (40, 32, 8, 128) if case == "mixed_d128" else (24, 16, 8, 64)
        lens = [int(rng.choice([0, 1, 15, 16, 17, 129, 1000, 3000])) for _ in range(B)]
        max_ctx = 3000
    else:
        B, Hq, Hkv, D = 200, 4, 1, 128
        lens = [int(x) for x in rng.integers(1, 6, size=B)]
        lens[77] = 8000
        max_ctx = 8000
    size = sum(-(-max(n, 1) // 16) * 16 for n in lens) + 64
    st = W.make_decode_step(lens=lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_layers=1, size=size,
                            page_size=16, seed=int(rng.integers(1 << 30)), max_ctx=max_ctx, device="cuda")
    # requests of length 0 have no new token: store the others' only
    nz = torch.tensor([i for i, n in enumerate(lens) if n > 0], dtype=torch.long)
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    k_new, v_new, loc = st.k_new[nz].contiguous(), st.v_new[nz].contiguous(), st.loc[nz.to(st.loc.device)].contiguous()
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, 0, k_new, v_new, loc)
    kb, vb = oracle.kv_store(kb0, vb0, 0, bits(k_new), bits(v_new), npy(loc))
    ref = _oracle_full(st, kb, vb)
    ws = _ws(B, Hq, Hkv, D, max_splits)
    out1, _ = _decode(st, max_splits=max_splits, ws=ws)
    assert_attention_close(npy(out1.float()), ref, f"balanced plan {case}")
    out2, _ = _decode(st, max_splits=max_splits, ws=ws)
    assert torch.equal(out1, out2)
    assert api.pa_get_error(ws) == 0


def test_bad_slot_sets_error_and_is_skipped():
    st = W.make_decode_step(lens=[40, 40], n_q_heads=8, n_kv_heads=2, head_dim=64, n_layers=1, size=256,
                            page_size=16, seed=8, device="cuda")
    kb, vb = _store_raw(st)
    row = int(st.kv.req_pool_indices[1])
    bad = st.kv.req_to_token.clone()
    bad[row, 5] = 10 ** 6
    out = torch.empty_like(st.q)
    ws = _ws(2, 8, 2, 64)
    api.pa_paged_decode_attn(st.q, st.kv.k_buf, st.kv.v_buf, 0, bad, st.kv.req_pool_indices, st.kv.seq_lens,
                             st.scale, ws, MAX_SPLITS, out)
    assert api.pa_get_error(ws) & api.DEVERR_SLOT
    ref = _oracle_full(st, kb, vb)
    assert_attention_close(npy(out.float())[0], ref[0], "untouched request")
    # request 1 equals attention over its other 39 tokens
    r2t = npy(st.kv.req_to_token).copy()
    keep = [j for j in range(40) if j != 5]
    r2t[row, :39] = r2t[row, keep]
    ref1 = oracle.decode(bits(st.q), kb, vb, 0, r2t, npy(st.kv.req_pool_indices), np.array([40, 39], np.int32),
                         st.scale)
    assert_attention_close(npy(out.float())[1], ref1[1], "skipped slot")
    assert np.isfinite(npy(out.float())).all()


# ------------------------------------------------------- full-size configs

@pytest.mark.parametrize("seq_len", [1024, 2048, 4096, 8192, 16384, 32768])
def test_config2_full_size(seq_len):
    """B=1, Hq=32, Hkv=8, D=128, [32, 65536, 8, 128] buffers, layer 17, page 16."""
    st = W.config2(seq_len, device="cuda", fill_layers=[17])
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    out, ws = _decode(st)
    k, v, r2t, rows, lens = compact_requests(st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                             st.kv.req_pool_indices, st.kv.seq_lens, [0])
    # the new token's row in the compact copy came from the device store: rebuild it from the inputs
    newpos = int(lens[0]) - 1
    k[0, r2t[0, newpos]] = bits(st.k_new)[0]
    v[0, r2t[0, newpos]] = bits(st.v_new)[0]
    ref = oracle.decode(bits(st.q), k, v, 0, r2t, rows, lens, st.scale)
    assert_attention_close(npy(out.float()), ref, f"config 2 seq {seq_len}")
    assert api.pa_get_error(ws) == 0


def test_config3_full_size():
    """B=32 ragged decode with 4 groups of 8 sharing a 1024-token prefix."""
    st = W.config3(device="cuda")
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    out, ws = _decode(st)
    B = st.q.shape[0]
    k, v, r2t, rows, lens = compact_requests(st.kv.k_buf, st.kv.v_buf, 0, st.kv.req_to_token,
                                             st.kv.req_pool_indices, st.kv.seq_lens, range(B))
    _restore_new_rows(st, k, v, r2t, lens, range(B))
    ref = oracle.decode(bits(st.q), k, v, 0, r2t, rows, lens, st.scale)
    assert_attention_close(npy(out.float()), ref, "config 3")
    assert api.pa_get_error(ws) == 0


def test_config5_full_size_sampled():
    """B=256, Hq=64, Hkv=8, page 1, 16M-slot buffers; oracle on sampled requests."""
    st = W.config5(device="cuda")
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, 0, st.k_new, st.v_new, st.loc)
    out, ws = _decode(st)
    lens = npy(st.kv.seq_lens)
    rng = np.random.default_rng(0)
    reqs = sorted(set([int(np.argmax(lens)), int(np.argmin(lens))] + rng.choice(256, 10, replace=False).tolist()))
    k, v, r2t, rows, slens = compact_requests(st.kv.k_buf, st.kv.v_buf, 0, st.kv.req_to_token,
                                              st.kv.req_pool_indices, st.kv.seq_lens, reqs)
    _restore_new_rows(st, k, v, r2t, slens, reqs)
    ref = oracle.decode(bits(st.q)[reqs], k, v, 0, r2t, rows, slens, st.scale)
    assert_attention_close(npy(out.float())[reqs], ref, "config 5 sampled")
    assert api.pa_get_error(ws) == 0
    assert torch.isfinite(out.float()).all()


def _restore_new_rows(st, k, v, r2t, lens, reqs):
    """Compact copies read the new tokens' rows back from the device: overwrite
    them with the step's inputs so the oracle sees only generator data."""
    kn, vn = bits(st.k_new), bits(st.v_new)
    for i, b in enumerate(reqs):
        n = int(lens[i])
        if n > 0:
            k[0, r2t[i, n - 1]] = kn[b]
            v[0, r2t[i, n - 1]] = vn[b]
