"""GPU parity of the e4m3 KV cache: the quantising store (bit-exact against
the oracle) and decode attention over it (|gpu - ref| <= 1e-2 + 1e-2 |ref|
against the oracle's float64 attention on the dequantised cache).

Inputs: the bf16 caches of the decode tests, quantised as a whole by the
library's store with per-(layer, kv head) scales near amax / 448, so the
bytes span the whole e4m3 range.  The oracle quantises the same bf16 values
on the host; both caches must agree byte for byte (NaN canaries: any NaN
code, since the NaN's sign is not part of the format's contract).
"""
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


def _scales(n_layers, Hkv, seed):
    g = np.random.default_rng(seed)
    return (torch.from_numpy((g.uniform(0.8, 1.25, (n_layers, Hkv)) * 4.5 / 448).astype(np.float32)),
            torch.from_numpy((g.uniform(0.8, 1.25, (n_layers, Hkv)) * 4.5 / 448).astype(np.float32)))


def _assert_bytes_equal(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    nan_w = (want & 0x7F) == 0x7F
    assert np.array_equal((got & 0x7F) == 0x7F, nan_w), f"{what}: NaN codes differ"
    bad = (got != want) & ~nan_w
    assert not bad.any(), f"{what}: {int(bad.sum())} bytes differ, first at {np.argwhere(bad)[0]}"


def _quantise_cache(kv, ks, vs):
    """Whole bf16 cache -> e4m3 on the device (library store, every slot of
    every layer) and on the host (oracle); returns device and host buffers."""
    n_layers, size, Hkv, D = kv.k_buf.shape
    k8 = torch.zeros((n_layers, size, Hkv, D), dtype=torch.uint8, device="cuda")
    v8 = torch.zeros_like(k8)
    ksd, vsd = ks.cuda(), vs.cuda()
    loc = torch.arange(size, dtype=torch.int32, device="cuda")
    kh, vh = np.zeros(k8.shape, np.uint8), np.zeros(v8.shape, np.uint8)
    for l in range(n_layers):
        api.pa_kv_store_fp8(k8, v8, l, kv.k_buf[l], kv.v_buf[l], loc, ksd, vsd)
        kh, vh = oracle.kv_store_fp8(kh, vh, l, bits(kv.k_buf[l]), bits(kv.v_buf[l]), npy(loc), npy(ks), npy(vs))
    torch.cuda.synchronize()
    _assert_bytes_equal(npy(k8), kh, "K cache")
    _assert_bytes_equal(npy(v8), vh, "V cache")
    return k8, v8, ksd, vsd, kh, vh


@pytest.mark.parametrize("Hkv,D", [(4, 64), (8, 128)])
def test_store_fp8_bit_exact_with_saturation_and_bad_slot(Hkv, D):
    g = W.generator(31 + D)
    n_layers, size, T = 2, 2048, 300
    k8 = torch.randint(0, 0x7E, (n_layers, size, Hkv, D), generator=g, dtype=torch.uint8).cuda()
    v8 = torch.randint(0, 0x7E, (n_layers, size, Hkv, D), generator=g, dtype=torch.uint8).cuda()
    k_new = (W.bf16_normal((T, Hkv, D), g) * 60).cuda()   # tails beyond 448 * scale saturate
    v_new = W.bf16_normal((T, Hkv, D), g).cuda()
    k_new[0, 0, :4] = torch.tensor([0.0, -0.0, 1e30, -1e30], dtype=torch.bfloat16)
    ks, vs = _scales(n_layers, Hkv, D)
    loc = torch.randperm(size, generator=g)[:T].to(torch.int32)
    kh, vh = oracle.kv_store_fp8(npy(k8), npy(v8), 1, bits(k_new), bits(v_new), npy(loc), npy(ks), npy(vs))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_kv_store_fp8(k8, v8, 1, k_new, v_new, loc.cuda(), ks.cuda(), vs.cuda(), err)
    torch.cuda.synchronize()
    _assert_bytes_equal(npy(k8), kh, "K")
    _assert_bytes_equal(npy(v8), vh, "V")
    assert api.pa_get_error_word(err) == 0
    # an out-of-range slot is skipped and flagged; the other tokens are written
    loc2 = torch.randperm(size, generator=g)[:8].to(torch.int32)
    loc2[3] = size
    before = npy(k8).copy()
    api.pa_kv_store_fp8(k8, v8, 0, k_new[:8], v_new[:8], loc2.cuda(), ks.cuda(), vs.cuda(), err)
    torch.cuda.synchronize()
    assert api.pa_get_error_word(err) & api.DEVERR_SLOT
    keep = np.r_[0:3, 4:8]
    want, _ = oracle.kv_store_fp8(before, npy(v8), 0, bits(k_new[:8])[keep], bits(v_new[:8])[keep],
                                  npy(loc2)[keep], npy(ks), npy(vs))
    _assert_bytes_equal(npy(k8), want, "K after a bad slot")


def _decode_fp8(st, k8, v8, ksd, vsd, max_splits=MAX_SPLITS):
    B, Hq, D = st.q.shape
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, k8.shape[2], D, max_splits))
    out = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn_fp8(st.q, k8, v8, st.layer, st.kv.req_to_token, st.kv.req_pool_indices,
                                 st.kv.seq_lens, st.scale, ksd, vsd, ws, max_splits, out)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    return out, ws


@pytest.mark.parametrize("Hq,Hkv,D,page", [(8, 2, 64, 16), (32, 8, 128, 16), (64, 8, 128, 1), (32, 2, 128, 4)])
def test_decode_fp8_ragged_batch(Hq, Hkv, D, page):
    """Store the step's new token into the fp8 cache, then decode; lengths
    around the tile (16) and split (64 .. 1024) boundaries, G = 4, 8, 16."""
    lens = [1, 16, 17, 64, 65, 300, 1024, 1025, 2100]
    st = W.make_decode_step(lens=lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_layers=2, size=8192,
                            page_size=page, seed=Hq * 5 + D + page, layer=1, req_rows=12, max_ctx=2200,
                            device="cuda")
    ks, vs = _scales(2, Hkv, Hq + D)
    k8, v8, ksd, vsd, kh, vh = _quantise_cache(st.kv, ks, vs)
    api.pa_kv_store_fp8(k8, v8, st.layer, st.k_new, st.v_new, st.loc, ksd, vsd)
    kh, vh = oracle.kv_store_fp8(kh, vh, st.layer, bits(st.k_new), bits(st.v_new), npy(st.loc), npy(ks), npy(vs))
    out, _ = _decode_fp8(st, k8, v8, ksd, vsd)
    ref = oracle.decode_fp8(bits(st.q), kh, vh, st.layer, npy(st.kv.req_to_token), npy(st.kv.req_pool_indices),
                            npy(st.kv.seq_lens), st.scale, npy(ks), npy(vs))
    assert_attention_close(npy(out.float()), ref, f"fp8 decode Hq={Hq} Hkv={Hkv} D={D}")


def test_decode_fp8_long_context_splits_deterministic_and_empty():
    """One 30K-token request (many splits), a 0-token and a 1-token request:
    sampled heads against the oracle, zeros for the empty request, and two
    calls bit-identical."""
    lens = [30000, 0, 1]
    st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=1, size=40000,
                            page_size=16, seed=77, layer=0, req_rows=4, max_ctx=30016, device="cuda")
    ks, vs = _scales(1, 8, 3)
    k8, v8, ksd, vsd, kh, vh = _quantise_cache(st.kv, ks, vs)
    has = [0, 2]   # the empty request has no token to store
    api.pa_kv_store_fp8(k8, v8, 0, st.k_new[has].contiguous(), st.v_new[has].contiguous(),
                        st.loc[has].contiguous(), ksd, vsd)
    kh, vh = oracle.kv_store_fp8(kh, vh, 0, bits(st.k_new)[has], bits(st.v_new)[has], npy(st.loc)[has],
                                 npy(ks), npy(vs))
    out1, _ = _decode_fp8(st, k8, v8, ksd, vsd)
    out2, _ = _decode_fp8(st, k8, v8, ksd, vsd)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.count_nonzero(out1[1]) == 0
    sel_b = np.array([0, 0, 0, 0, 2, 2], np.int32)
    sel_h = np.array([0, 9, 22, 31, 5, 30], np.int32)
    ref = oracle.decode_fp8(bits(st.q), kh, vh, 0, npy(st.kv.req_to_token), npy(st.kv.req_pool_indices),
                            npy(st.kv.seq_lens), st.scale, npy(ks), npy(vs), sel=(sel_b, sel_h))
    assert_attention_close(npy(out1.float())[sel_b, sel_h], ref, "fp8 decode 30K")


@pytest.mark.parametrize("seq_len", [4096, 32768])
def test_config2_full_size_fp8(seq_len):
    """The bench's e4m3 sweep configuration: the [32, 65536, 8, 128] cache
    quantised by the library's store (layer 17), the step's new token stored,
    B=1 decode with the bench's split cap.  The request's slots are compared
    byte for byte with the oracle's quantisation of the generator's bf16 rows
    (compacted on the host, the new row taken from the step's inputs), and the
    output with the oracle's attention over those bytes."""
    st = W.config2(seq_len, device="cuda", fill_layers=[17])
    dev = st.q.device
    n_layers, size, Hkv, D = st.kv.k_buf.shape
    ks, vs = _scales(n_layers, Hkv, seq_len)
    ksd, vsd = ks.to(dev), vs.to(dev)
    k8 = torch.zeros((n_layers, size, Hkv, D), dtype=torch.uint8, device=dev)
    v8 = torch.zeros_like(k8)
    every = torch.arange(size, dtype=torch.int32, device=dev)
    api.pa_kv_store_fp8(k8, v8, st.layer, st.kv.k_buf[st.layer], st.kv.v_buf[st.layer], every, ksd, vsd)
    api.pa_kv_store_fp8(k8, v8, st.layer, st.k_new, st.v_new, st.loc, ksd, vsd)
    out, _ = _decode_fp8(st, k8, v8, ksd, vsd)
    # host side: the request's rows in sorted-slot order, from generator data only
    row = int(st.kv.req_pool_indices[0])
    slots = st.kv.req_to_token[row, :seq_len].long()
    uniq, inv = torch.unique(slots, return_inverse=True)
    kb = bits(st.kv.k_buf[st.layer][uniq])
    vb = bits(st.kv.v_buf[st.layer][uniq])
    new = int(inv[seq_len - 1])
    kb[new], vb[new] = bits(st.k_new)[0], bits(st.v_new)[0]
    U = uniq.numel()
    l_ks, l_vs = npy(ks)[st.layer][None], npy(vs)[st.layer][None]
    kh, vh = oracle.kv_store_fp8(np.zeros((1, U, Hkv, D), np.uint8), np.zeros((1, U, Hkv, D), np.uint8), 0,
                                 kb, vb, np.arange(U, dtype=np.int32), l_ks, l_vs)
    _assert_bytes_equal(npy(k8[st.layer][uniq]), kh[0], "K rows of the request")
    _assert_bytes_equal(npy(v8[st.layer][uniq]), vh[0], "V rows of the request")
    r2t = npy(inv).astype(np.int32)[None]
    ref = oracle.decode_fp8(bits(st.q), kh, vh, 0, r2t, np.zeros(1, np.int32), np.array([seq_len], np.int32),
                            st.scale, l_ks, l_vs)
    assert_attention_close(npy(out.float()), ref, f"fp8 config 2 seq {seq_len}")


# ------------------------------------------------------------ fp8 prefill

def _prefill_fp8_case(new, pre, Hq, Hkv, D, page, seed, size=8192):
    """A packed prefill batch over an e4m3 cache: the generator's bf16 cache
    quantised whole by the library's store (and by the oracle on the host),
    then the new tokens' K/V stored quantised at their slots on both sides."""
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D,
                              size=size, page_size=page, seed=seed, req_rows=len(new) + 3, device="cuda")
    ks, vs = _scales(1, Hkv, seed)
    k8, v8, ksd, vsd, kh, vh = _quantise_cache(pb.kv, ks, vs)
    api.pa_kv_store_fp8(k8, v8, pb.layer, pb.k_new, pb.v_new, pb.loc, ksd, vsd)
    kh, vh = oracle.kv_store_fp8(kh, vh, pb.layer, bits(pb.k_new), bits(pb.v_new), npy(pb.loc), npy(ks), npy(vs))
    return pb, k8, v8, ksd, vsd, kh, vh, ks, vs


def _prefill_fp8(pb, k8, v8, ksd, vsd, ws=None):
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes()) if ws is None else ws
    out = torch.full_like(pb.q, float("nan"))
    api.pa_paged_prefill_attn_fp8(pb.q, k8, v8, pb.layer, pb.qo_indptr, pb.kv_indptr, pb.kv.req_to_token,
                                  pb.kv.req_pool_indices, pb.scale, ksd, vsd, ws, out)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    return out, ws


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("D,page", [(128, 16), (64, 1)])
def test_prefill_fp8_ragged(G, D, page):
    """Ragged prompts with and without cached prefixes, lengths around the
    128-row q and kv tile edges, G = 1 .. 16, head_dim 64 and 128, page
    sizes 16 (box gathers) and 1 (row gathers)."""
    new, pre = [1, 31, 130, 7, 300, 128], [0, 5, 300, 17, 1000, 129]
    pb, k8, v8, ksd, vsd, kh, vh, ks, vs = _prefill_fp8_case(new, pre, 2 * G, 2, D, page, seed=G * 13 + D + page)
    out, _ = _prefill_fp8(pb, k8, v8, ksd, vsd)
    ref = oracle.prefill_fp8(bits(pb.q), kh, vh, pb.layer, npy(pb.qo_indptr), npy(pb.kv_indptr),
                             npy(pb.kv.req_to_token), npy(pb.kv.req_pool_indices), pb.scale, npy(ks), npy(vs))
    assert_attention_close(npy(out.float()), ref, f"fp8 prefill G={G} D={D} page={page}")


def test_prefill_fp8_config4_shape_sampled_and_deterministic():
    """Config 4's prompt lengths, heads and cache over an e4m3 copy: every
    head of the first, last and 4 random rows of each request against the
    oracle, and two calls bit-identical."""
    pb = W.config4(device="cuda")
    ks, vs = _scales(1, 8, 4)
    k8, v8, ksd, vsd, kh, vh = _quantise_cache(pb.kv, ks, vs)
    api.pa_kv_store_fp8(k8, v8, pb.layer, pb.k_new, pb.v_new, pb.loc, ksd, vsd)
    kh, vh = oracle.kv_store_fp8(kh, vh, pb.layer, bits(pb.k_new), bits(pb.v_new), npy(pb.loc), npy(ks), npy(vs))
    out1, ws = _prefill_fp8(pb, k8, v8, ksd, vsd)
    out2, _ = _prefill_fp8(pb, k8, v8, ksd, vsd, ws=ws)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    qo = npy(pb.qo_indptr)
    rng = np.random.default_rng(44)
    rows = []
    for r in range(len(pb.new_lens)):
        rows += [qo[r], qo[r + 1] - 1] + rng.integers(qo[r], qo[r + 1], 4).tolist()
    rows = sorted(set(int(x) for x in rows))
    Hq = pb.q.shape[1]
    st = np.repeat(np.array(rows, np.int32), Hq)
    sh = np.tile(np.arange(Hq, dtype=np.int32), len(rows))
    ref = oracle.prefill_fp8(bits(pb.q), kh, vh, pb.layer, qo, npy(pb.kv_indptr), npy(pb.kv.req_to_token),
                             npy(pb.kv.req_pool_indices), pb.scale, npy(ks), npy(vs), sel=(st, sh))
    assert_attention_close(npy(out1.float())[st, sh], ref, "fp8 prefill, config 4 sampled")
