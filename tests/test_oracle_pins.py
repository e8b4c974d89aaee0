"""Pins for the float64 oracle, checked against things other than itself.

Each test ties an oracle function to a hand-worked value (tests/golden), a
library routine on a special case (torch's scaled_dot_product_attention in
float64, numpy complex multiplication, numpy fancy indexing, torch's fp32->bf16
conversion), a closed form, or an invariant that a plausible slip in the
oracle (a wrong GQA head, a dropped key, a transposed pair, a misaligned causal
mask) would break.  No GPU needed.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_188_gb300 import workloads as W


def bits(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _scale(v):
    return math.log(3.0) / 2 if v == "ln3/2" else float(v)


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "bf16_rounding.json")))
    for c in g["cases"]:
        got = int(oracle.f64_to_bf16(np.array([c["value"]]))[0])
        assert got == int(c["bits"], 16), (c["x"], hex(got))


def test_bf16_rounding_matches_torch_on_fp32_values():
    # for values that are exact fp32 numbers, torch's fp32->bf16 conversion is a
    # single round-to-nearest-even: the oracle's double->bf16 must agree.
    g = torch.Generator().manual_seed(11)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 20)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-40, -3e-39, 3.0e38, -3.3e38])])
    want = bits(x.to(torch.bfloat16))
    got = oracle.f64_to_bf16(x.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, want)


def test_bf16_widening_exact():
    b = np.array([0x3F80, 0xC000, 0x7F80, 0x0001, 0x3DCD], dtype=np.uint16)
    np.testing.assert_array_equal(oracle.bf16_to_f64(b), [1.0, -2.0, np.inf, 2.0 ** -133, 0.10009765625])


# ------------------------------------------------------------------ RoPE

def test_rope_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "rope_hand.json")))
    cos = np.array(g["cos"], dtype=np.float32)
    sin = np.array(g["sin"], dtype=np.float32)
    for c in g["cases"]:
        x = torch.tensor([[c["x"]]], dtype=torch.bfloat16)
        yb, yf = oracle.rope(bits(x), np.array([c["pos"]], np.int32), cos, sin)
        np.testing.assert_array_equal(yf[0, 0], c["expect"])
        np.testing.assert_array_equal(oracle.bf16_to_f64(yb[0, 0]), c["expect"])


def test_rope_matches_complex_multiplication():
    # interleaved pairs are complex numbers x0 + i x1 multiplied by c + i s
    T, H, D = 37, 3, 64
    g = W.generator(5)
    x = W.bf16_normal((T, H, D), g)
    cos, sin = W.rope_tables(4096, D)
    pos = torch.randint(0, 4096, (T,), generator=g, dtype=torch.int32)
    _, yf = oracle.rope(bits(x), pos.numpy(), cos.numpy(), sin.numpy())
    xc = f64(x)[..., 0::2] + 1j * f64(x)[..., 1::2]
    rot = (cos.double().numpy()[pos.numpy()] + 1j * sin.double().numpy()[pos.numpy()])[:, None, :]
    want = xc * rot
    np.testing.assert_allclose(yf[..., 0::2], want.real, rtol=0, atol=1e-13)
    np.testing.assert_allclose(yf[..., 1::2], want.imag, rtol=0, atol=1e-13)


def test_rope_angle_closed_form_and_norm():
    # unit vector e_{2i} at position p rotates to (cos, sin)(p * theta^(-2i/D))
    D = 128
    cos, sin = W.rope_tables(W.ROPE_MAX_POS, D)
    for p in [0, 1, 7, 1000, 32767]:
        x = torch.zeros(1, D // 2, D, dtype=torch.bfloat16)
        for i in range(D // 2):
            x[0, i, 2 * i] = 1.0
        _, yf = oracle.rope(bits(x), np.array([p], np.int32), cos.numpy(), sin.numpy())
        for i in [0, 1, 17, 63]:
            ang = p * 10000.0 ** (-2.0 * i / D)
            assert abs(yf[0, i, 2 * i] - math.cos(ang)) < 2e-7
            assert abs(yf[0, i, 2 * i + 1] - math.sin(ang)) < 2e-7
            others = np.delete(yf[0, i], [2 * i, 2 * i + 1])
            assert not others.any()
    # pair norms are preserved up to the fp32 table's rounding
    g = W.generator(6)
    x = W.bf16_normal((50, 4, D), g)
    pos = torch.randint(0, W.ROPE_MAX_POS, (50,), generator=g, dtype=torch.int32)
    _, yf = oracle.rope(bits(x), pos.numpy(), cos.numpy(), sin.numpy())
    n0 = f64(x)[..., 0::2] ** 2 + f64(x)[..., 1::2] ** 2
    n1 = yf[..., 0::2] ** 2 + yf[..., 1::2] ** 2
    np.testing.assert_allclose(n1, n0, rtol=5e-7, atol=1e-30)


def test_rope_composes_rotations():
    # R(b) applied to R(a) x equals R(a+b) x, to the fp32 table's accuracy
    D = 64
    cos, sin = W.rope_tables(W.ROPE_MAX_POS, D)
    g = W.generator(8)
    x = W.bf16_normal((1, 1, D), g)
    a, b = 123, 4567
    _, ya = oracle.rope(bits(x), np.array([a], np.int32), cos.numpy(), sin.numpy())
    # apply R(b) to the float64 result by the same pair rule, via complex numbers
    ya_c = ya[..., 0::2] + 1j * ya[..., 1::2]
    yab = ya_c * (cos.double().numpy()[b] + 1j * sin.double().numpy()[b])
    _, y_sum = oracle.rope(bits(x), np.array([a + b], np.int32), cos.numpy(), sin.numpy())
    np.testing.assert_allclose(y_sum[..., 0::2], yab.real, atol=2e-6)
    np.testing.assert_allclose(y_sum[..., 1::2], yab.imag, atol=2e-6)


def test_rope_rejects_bad_position():
    cos, sin = W.rope_tables(16, 8)
    x = torch.zeros(1, 1, 8, dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.rope(bits(x), np.array([16], np.int32), cos.numpy(), sin.numpy())


# -------------------------------------------------------------- kv store

def test_kv_store_matches_fancy_indexing():
    g = W.generator(9)
    kb = W.nan_filled((3, 64, 2, 8))
    vb = W.nan_filled((3, 64, 2, 8))
    kb[1, :10] = W.bf16_normal((10, 2, 8), g)
    kn = W.bf16_normal((7, 2, 8), g)
    vn = W.bf16_normal((7, 2, 8), g)
    loc = torch.randperm(64, generator=g)[:7].to(torch.int32)
    k2, v2 = oracle.kv_store(bits(kb), bits(vb), 1, bits(kn), bits(vn), loc.numpy())
    kw, vw = bits(kb).copy(), bits(vb).copy()
    kw[1, loc.numpy()] = bits(kn)
    vw[1, loc.numpy()] = bits(vn)
    np.testing.assert_array_equal(k2, kw)
    np.testing.assert_array_equal(v2, vw)
    with pytest.raises(oracle.OracleError):
        oracle.kv_store(bits(kb), bits(vb), 1, bits(kn), bits(vn), np.array([0, 1, 2, 3, 4, 5, 64], np.int32))


# ------------------------------------------------------------- attention

def _sdpa_f64(q, k, v, scale, mask=None, causal=False):
    """torch's float64 scaled_dot_product_attention, one head at a time.
    q [n, D], k/v [m, D]."""
    return F.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
        torch.from_numpy(v)[None, None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None],
        is_causal=causal, scale=scale)[0, 0].numpy()


def _decode_args(st: W.DecodeStep, kb=None, vb=None):
    return (bits(st.q), bits(st.kv.k_buf if kb is None else kb), bits(st.kv.v_buf if vb is None else vb),
            st.layer, st.kv.req_to_token.numpy(), st.kv.req_pool_indices.numpy(),
            st.kv.seq_lens.numpy(), st.scale)


def _fill_new_token(st: W.DecodeStep):
    """Put the step's raw new K/V at their slots (no rotary), so the cache is complete."""
    kb, vb = oracle.kv_store(bits(st.kv.k_buf), bits(st.kv.v_buf), st.layer, bits(st.k_new),
                             bits(st.v_new), st.loc.numpy())
    return kb, vb


@pytest.mark.parametrize("Hq,Hkv,D,page,lens", [
    (4, 4, 8, 4, [5, 1, 9]), (4, 2, 8, 1, [3, 7]), (8, 2, 16, 4, [13, 16, 2]),
    (6, 3, 4, 2, [4]), (16, 2, 32, 16, [40, 17])])
def test_decode_matches_library_sdpa(Hq, Hkv, D, page, lens):
    st = W.make_decode_step(lens=lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_layers=2,
                            size=128, page_size=page, seed=sum(lens) + Hq, layer=1,
                            req_rows=len(lens) + 3, max_ctx=max(lens) + 5)
    kb, vb = _fill_new_token(st)
    out = oracle.decode(*_decode_args(st, kb, vb))
    G = Hq // Hkv
    qf = oracle.bf16_to_f64(bits(st.q))
    kf = oracle.bf16_to_f64(kb)
    vf = oracle.bf16_to_f64(vb)
    for b, n in enumerate(lens):
        row = int(st.kv.req_pool_indices[b])
        slots = st.kv.req_to_token[row, :n].numpy()
        for hq in range(Hq):
            ref = _sdpa_f64(qf[b, hq][None], kf[1, slots, hq // G], vf[1, slots, hq // G], st.scale)
            np.testing.assert_allclose(out[b, hq], ref[0], rtol=1e-12, atol=1e-12)


def test_attention_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "attention_hand.json")))
    for c in g["decode"]:
        D, Hq, Hkv = c["D"], c["Hq"], c["Hkv"]
        K = torch.tensor(c["K"], dtype=torch.bfloat16)
        V = torch.tensor(c["V"], dtype=torch.bfloat16)
        n = K.shape[0]
        size = 8
        kb = W.nan_filled((1, size, Hkv, D))
        vb = W.nan_filled((1, size, Hkv, D))
        slots = [5, 2, 7, 0][:n]
        kb[0, slots, 0] = K
        vb[0, slots, 0] = V
        r2t = np.full((2, 4), -3, np.int32)
        r2t[1, :n] = slots
        q = torch.tensor(c["q"], dtype=torch.bfloat16)[None]
        out = oracle.decode(bits(q), bits(kb), bits(vb), 0, r2t, np.array([1], np.int32),
                            np.array([n], np.int32), _scale(c["scale"]))
        np.testing.assert_allclose(out[0], c["expect"], rtol=1e-14, atol=1e-14, err_msg=c["name"])
    for c in g["prefill"]:
        D, p, n = c["D"], c["prefix"], c["new"]
        size = 8
        kb = W.nan_filled((1, size, 1, D))
        vb = W.nan_filled((1, size, 1, D))
        slots = [6, 1, 3]
        kb[0, slots, 0] = torch.tensor(c["K"], dtype=torch.bfloat16)
        vb[0, slots, 0] = torch.tensor(c["V"], dtype=torch.bfloat16)
        r2t = np.array([slots + [-1]], np.int32)
        q = torch.tensor(c["q"], dtype=torch.bfloat16)[:, None, :]
        out = oracle.prefill(bits(q), bits(kb), bits(vb), 0, np.array([0, n], np.int32),
                             np.array([0, p + n], np.int32), r2t, np.array([0], np.int32),
                             _scale(c["scale"]))
        np.testing.assert_allclose(out[:, 0], c["expect"], rtol=1e-14, atol=1e-14, err_msg=c["name"])


def test_decode_closed_forms():
    st = W.make_decode_step(lens=[9, 4], n_q_heads=4, n_kv_heads=2, head_dim=8, n_layers=1,
                            size=64, page_size=4, seed=21)
    kb, vb = _fill_new_token(st)
    # scale 0 -> uniform weights -> the mean of the request's V rows
    args = list(_decode_args(st, kb, vb))
    args[-1] = 0.0
    out = oracle.decode(*args)
    vf = oracle.bf16_to_f64(vb)
    for b, n in enumerate([9, 4]):
        row = int(st.kv.req_pool_indices[b])
        slots = st.kv.req_to_token[row, :n].numpy()
        for hq in range(4):
            np.testing.assert_allclose(out[b, hq], vf[0, slots, hq // 2].mean(0), rtol=1e-13, atol=1e-14)
    # constant V rows -> that constant, whatever the scores
    vconst = vb.copy()
    vconst[...] = bits(torch.tensor(1.75, dtype=torch.bfloat16).reshape(1))[0]
    out = oracle.decode(*_decode_args(st, kb, vconst))
    np.testing.assert_allclose(out, 1.75, rtol=1e-14)
    # an empty request gives zeros
    args = list(_decode_args(st, kb, vb))
    args[6] = np.array([0, 4], np.int32)
    out = oracle.decode(*args)
    assert not out[0].any()


def test_decode_invariant_to_page_placement_and_stale_entries():
    st = W.make_decode_step(lens=[30, 11, 25], n_q_heads=8, n_kv_heads=2, head_dim=16, n_layers=1,
                            size=256, page_size=4, seed=31, req_rows=5, max_ctx=40)
    kb, vb = _fill_new_token(st)
    base = oracle.decode(*_decode_args(st, kb, vb))
    # move every slot to a new physical place and rewrite the table accordingly
    perm = np.random.default_rng(3).permutation(256)
    kb2, vb2 = np.empty_like(kb), np.empty_like(vb)
    kb2[:, perm] = kb
    vb2[:, perm] = vb
    r2t = st.kv.req_to_token.numpy().copy()
    r2t2 = r2t.copy()
    ok = (r2t >= 0) & (r2t < 256)
    r2t2[ok] = perm[r2t[ok]]
    # garbage past each request's length must not matter
    for b, n in enumerate([30, 11, 25]):
        r2t2[int(st.kv.req_pool_indices[b]), n:] = -12345
    out = oracle.decode(bits(st.q), kb2, vb2, 0, r2t2, st.kv.req_pool_indices.numpy(),
                        st.kv.seq_lens.numpy(), st.scale)
    np.testing.assert_array_equal(out, base)


def test_decode_gqa_equals_replicated_mha():
    # Hq=8 over Hkv=2 must equal Hq=8 over 8 kv heads where kv head j is a copy
    # of original head j // 4 (contiguous grouping)
    st = W.make_decode_step(lens=[12, 7], n_q_heads=8, n_kv_heads=2, head_dim=8, n_layers=1,
                            size=64, page_size=2, seed=41)
    kb, vb = _fill_new_token(st)
    out_gqa = oracle.decode(*_decode_args(st, kb, vb))
    kb_rep = np.repeat(kb, 4, axis=2)
    vb_rep = np.repeat(vb, 4, axis=2)
    out_mha = oracle.decode(bits(st.q), kb_rep, vb_rep, 0, st.kv.req_to_token.numpy(),
                            st.kv.req_pool_indices.numpy(), st.kv.seq_lens.numpy(), st.scale)
    np.testing.assert_array_equal(out_gqa, out_mha)
    # and the grouping is not the interleaved one: head 1 differs from head 5's view
    assert not np.allclose(out_gqa[:, 1], out_gqa[:, 5])


def test_decode_selected_pairs_match_full():
    st = W.make_decode_step(lens=[12, 7, 3], n_q_heads=8, n_kv_heads=4, head_dim=8, n_layers=1,
                            size=64, page_size=2, seed=42)
    kb, vb = _fill_new_token(st)
    full = oracle.decode(*_decode_args(st, kb, vb))
    sb = np.array([2, 0, 1, 1], np.int32)
    sh = np.array([7, 0, 3, 4], np.int32)
    sel = oracle.decode(*_decode_args(st, kb, vb), sel=(sb, sh))
    np.testing.assert_array_equal(sel, full[sb, sh])


def _prefill_complete(pb: W.PrefillBatch):
    kb, vb = oracle.kv_store(bits(pb.kv.k_buf), bits(pb.kv.v_buf), pb.layer, bits(pb.k_new),
                             bits(pb.v_new), pb.loc.numpy())
    return kb, vb


def test_prefill_no_prefix_is_textbook_causal():
    pb = W.make_prefill_batch(new_lens=[23], prefix_lens=[0], n_q_heads=4, n_kv_heads=2, head_dim=16,
                              size=128, page_size=4, seed=51)
    kb, vb = _prefill_complete(pb)
    out = oracle.prefill(bits(pb.q), kb, vb, 0, pb.qo_indptr.numpy(), pb.kv_indptr.numpy(),
                         pb.kv.req_to_token.numpy(), pb.kv.req_pool_indices.numpy(), pb.scale)
    row = int(pb.kv.req_pool_indices[0])
    slots = pb.kv.req_to_token[row, :23].numpy()
    qf = oracle.bf16_to_f64(bits(pb.q))
    kf, vf = oracle.bf16_to_f64(kb), oracle.bf16_to_f64(vb)
    for hq in range(4):
        ref = _sdpa_f64(qf[:, hq], kf[0, slots, hq // 2], vf[0, slots, hq // 2], pb.scale, causal=True)
        np.testing.assert_allclose(out[:, hq], ref, rtol=1e-12, atol=1e-12)


def test_prefill_with_prefix_matches_masked_library_attention():
    new, pre = [5, 17, 1, 9], [11, 0, 6, 32]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=6, n_kv_heads=3, head_dim=8,
                              size=256, page_size=4, seed=52, req_rows=7)
    kb, vb = _prefill_complete(pb)
    out = oracle.prefill(bits(pb.q), kb, vb, 0, pb.qo_indptr.numpy(), pb.kv_indptr.numpy(),
                         pb.kv.req_to_token.numpy(), pb.kv.req_pool_indices.numpy(), pb.scale)
    qf = oracle.bf16_to_f64(bits(pb.q))
    kf, vf = oracle.bf16_to_f64(kb), oracle.bf16_to_f64(vb)
    t0 = 0
    for r, (n, p) in enumerate(zip(new, pre)):
        row = int(pb.kv.req_pool_indices[r])
        slots = pb.kv.req_to_token[row, :p + n].numpy()
        mask = np.arange(p + n)[None, :] <= (p + np.arange(n))[:, None]   # bottom-right aligned
        for hq in range(6):
            ref = _sdpa_f64(qf[t0:t0 + n, hq], kf[0, slots, hq // 2], vf[0, slots, hq // 2], pb.scale,
                            mask=mask)
            np.testing.assert_allclose(out[t0:t0 + n, hq], ref, rtol=1e-12, atol=1e-12)
        t0 += n


def test_prefill_last_row_equals_decode():
    new, pre = [7, 3, 12], [4, 20, 0]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=4, n_kv_heads=1, head_dim=8,
                              size=128, page_size=4, seed=53)
    kb, vb = _prefill_complete(pb)
    out = oracle.prefill(bits(pb.q), kb, vb, 0, pb.qo_indptr.numpy(), pb.kv_indptr.numpy(),
                         pb.kv.req_to_token.numpy(), pb.kv.req_pool_indices.numpy(), pb.scale)
    last = pb.qo_indptr.numpy()[1:] - 1
    qdec = bits(pb.q)[last]
    dec = oracle.decode(qdec, kb, vb, 0, pb.kv.req_to_token.numpy(), pb.kv.req_pool_indices.numpy(),
                        np.array([p + n for p, n in zip(pre, new)], np.int32), pb.scale)
    np.testing.assert_array_equal(out[last], dec)


def test_prefill_packing_is_per_request():
    # request r's rows do not depend on the other requests in the pack
    new, pre = [6, 4], [3, 9]
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=2, n_kv_heads=2, head_dim=8,
                              size=64, page_size=2, seed=54)
    kb, vb = _prefill_complete(pb)
    r2t, rpi = pb.kv.req_to_token.numpy(), pb.kv.req_pool_indices.numpy()
    out = oracle.prefill(bits(pb.q), kb, vb, 0, pb.qo_indptr.numpy(), pb.kv_indptr.numpy(), r2t, rpi,
                         pb.scale)
    alone = oracle.prefill(bits(pb.q)[6:], kb, vb, 0, np.array([0, 4], np.int32),
                           np.array([0, 13], np.int32), r2t, rpi[1:], pb.scale)
    np.testing.assert_array_equal(out[6:], alone)
    sel = oracle.prefill(bits(pb.q), kb, vb, 0, pb.qo_indptr.numpy(), pb.kv_indptr.numpy(), r2t, rpi,
                         pb.scale, sel=(np.array([9, 0], np.int32), np.array([1, 0], np.int32)))
    np.testing.assert_array_equal(sel, out[[9, 0], [1, 0]])


# ------------------------------------------------------- fp8 (e4m3) cache

def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    """torch's float32 -> float8_e4m3fn conversion (nearest, ties to even;
    NaN above 464, where rounding reaches 480 and the oracle saturates)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_e4m3_values(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_e4m3_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "e4m3_hand.json")))
    for c in g["decode"]:
        got = float(oracle.e4m3_to_f64(np.array([int(c["code"], 16)], np.uint8))[0])
        if c["value"] == "nan":
            assert math.isnan(got), c
        else:
            assert got == c["value"] and math.copysign(1, got) == math.copysign(1, c["value"]), (c, got)
    for c in g["encode"]:
        got = int(oracle.f32_to_e4m3(np.array([c["value"]], np.float32))[0])
        assert got == int(c["code"], 16), (c, hex(got))


def test_e4m3_values_match_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = _torch_e4m3_values(codes)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])
    assert np.isnan(ours[[0x7F, 0xFF]]).all() and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    assert np.signbit(ours[0x80]) and ours[0x80] == 0.0


def test_e4m3_encoding_matches_torch_up_to_464():
    g = np.random.default_rng(11)
    parts = [g.standard_normal(4000) * 2.0 ** k for k in range(-12, 9)]
    finite = _torch_e4m3_values(np.arange(256, dtype=np.uint8))
    finite = np.unique(finite[~np.isnan(finite)])
    mids = (finite[1:] + finite[:-1]) / 2          # every tie between neighbouring codes
    parts += [finite, mids, -mids, np.array([0.0, -0.0, 447.9, 463.9, 464.0, -464.0])]
    x = np.concatenate(parts).astype(np.float32)
    x = x[np.abs(x) <= 464]
    np.testing.assert_array_equal(oracle.f32_to_e4m3(x), _torch_e4m3(x))


def test_e4m3_saturates_and_round_trips():
    big = np.array([448.0, 464.5, 479.9, 480.0, 1000.0, 3.0e38, np.inf], np.float32)
    np.testing.assert_array_equal(oracle.f32_to_e4m3(big), np.full(7, 0x7E, np.uint8))
    np.testing.assert_array_equal(oracle.f32_to_e4m3(-big), np.full(7, 0xFE, np.uint8))
    assert oracle.f32_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    vals = oracle.e4m3_to_f64(codes).astype(np.float32)
    np.testing.assert_array_equal(oracle.f32_to_e4m3(vals), codes)


def test_kv_store_fp8_matches_torch_quantisation():
    g = W.generator(23)
    L, size, Hkv, D = 2, 48, 3, 16
    kb = np.full((L, size, Hkv, D), 0x7F, np.uint8)
    vb = np.full((L, size, Hkv, D), 0x7F, np.uint8)
    kn = W.bf16_normal((9, Hkv, D), g) * 40
    vn = W.bf16_normal((9, Hkv, D), g)
    kn[0, 0, :4] = torch.tensor([1e4, -1e4, 0.0, -0.0])   # saturating and signed-zero entries
    ks = np.array([[0.5, 0.03, 1.7], [0.25, 0.11, 3.0]], np.float32)
    vs = np.array([[0.01, 0.2, 0.007], [0.004, 0.09, 1.0]], np.float32)
    loc = torch.randperm(size, generator=g)[:9].numpy().astype(np.int32)
    k2, v2 = oracle.kv_store_fp8(kb, vb, 1, bits(kn), bits(vn), loc, ks, vs)
    kw, vw = kb.copy(), vb.copy()
    for new, sc, want in ((kn, ks, kw), (vn, vs, vw)):
        q = (new.float() / torch.from_numpy(sc[1])[None, :, None]).clamp(-448, 448)   # fp32 division
        want[1, loc] = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(k2, kw)
    np.testing.assert_array_equal(v2, vw)
    with pytest.raises(oracle.OracleError):
        oracle.kv_store_fp8(kb, vb, 1, bits(kn), bits(vn), np.r_[loc[:8], size].astype(np.int32), ks, vs)


def _fp8_step(lens, Hq, Hkv, D, page, seed):
    """A decode step over an fp8 cache: the bf16 cache of the same seed
    quantised with per-(layer, kv head) scales (by the oracle's store)."""
    st = W.make_decode_step(lens=lens, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D, n_layers=2, size=128,
                            page_size=page, seed=seed, layer=1, req_rows=len(lens) + 3, max_ctx=max(lens) + 5)
    kb, vb = _fill_new_token(st)
    rng = np.random.default_rng(seed)
    ks = (rng.uniform(0.5, 2.0, (2, Hkv)) / 112).astype(np.float32)
    vs = (rng.uniform(0.5, 2.0, (2, Hkv)) / 112).astype(np.float32)
    k8 = oracle.f32_to_e4m3(oracle.bf16_to_f64(kb).astype(np.float32) / ks[:, None, :, None])
    v8 = oracle.f32_to_e4m3(oracle.bf16_to_f64(vb).astype(np.float32) / vs[:, None, :, None])
    return st, k8, v8, ks, vs


@pytest.mark.parametrize("Hq,Hkv,D,page,lens", [
    (4, 4, 8, 4, [5, 1, 9]), (8, 2, 16, 1, [13, 7]), (16, 2, 32, 16, [40, 17])])
def test_decode_fp8_matches_library_sdpa_on_dequantised_cache(Hq, Hkv, D, page, lens):
    st, k8, v8, ks, vs = _fp8_step(lens, Hq, Hkv, D, page, seed=sum(lens) + D)
    out = oracle.decode_fp8(bits(st.q), k8, v8, 1, st.kv.req_to_token.numpy(), st.kv.req_pool_indices.numpy(),
                            st.kv.seq_lens.numpy(), st.scale, ks, vs)
    kf = _torch_e4m3_values(k8) * ks[:, None, :, None].astype(np.float64)
    vf = _torch_e4m3_values(v8) * vs[:, None, :, None].astype(np.float64)
    qf = oracle.bf16_to_f64(bits(st.q))
    G = Hq // Hkv
    for b, n in enumerate(lens):
        slots = st.kv.req_to_token[int(st.kv.req_pool_indices[b]), :n].numpy()
        for hq in range(Hq):
            ref = _sdpa_f64(qf[b, hq][None], kf[1, slots, hq // G], vf[1, slots, hq // G], st.scale)
            np.testing.assert_allclose(out[b, hq], ref[0], rtol=1e-12, atol=1e-12)


def test_decode_fp8_with_power_of_two_scales_equals_bf16_decode():
    # e4m3 values times 2^k are bf16 numbers, so the bf16 oracle on the
    # dequantised cache computes the same attention
    st, k8, v8, _, _ = _fp8_step([11, 30], 8, 2, 16, 4, seed=5)
    ks = np.array([[2.0 ** -5, 2.0 ** -7], [2.0 ** -6, 2.0 ** -4]], np.float32)
    vs = np.array([[2.0 ** -3, 1.0], [2.0 ** -8, 2.0 ** -6]], np.float32)
    kbf = oracle.f64_to_bf16(oracle.e4m3_to_f64(k8) * ks[:, None, :, None])
    vbf = oracle.f64_to_bf16(oracle.e4m3_to_f64(v8) * vs[:, None, :, None])
    args = (st.kv.req_to_token.numpy(), st.kv.req_pool_indices.numpy(), st.kv.seq_lens.numpy(), st.scale)
    ref = oracle.decode(bits(st.q), kbf, vbf, 1, *args)
    out = oracle.decode_fp8(bits(st.q), k8, v8, 1, *args, ks, vs)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-15)


def _fp8_prefill(new, pre, Hq, Hkv, D, page, seed, ks=None, vs=None):
    """A prefill batch over an fp8 cache: the complete bf16 cache (prefix +
    new tokens, stored by the oracle) quantised with per-(layer, kv head)
    scales by the oracle's encoder."""
    pb = W.make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=D,
                              size=256, page_size=page, seed=seed, req_rows=len(new) + 2)
    kb, vb = _prefill_complete(pb)
    rng = np.random.default_rng(seed)
    L = kb.shape[0]
    ks = (rng.uniform(0.5, 2.0, (L, Hkv)) / 112).astype(np.float32) if ks is None else ks
    vs = (rng.uniform(0.5, 2.0, (L, Hkv)) / 112).astype(np.float32) if vs is None else vs
    k8 = oracle.f32_to_e4m3(oracle.bf16_to_f64(kb).astype(np.float32) / ks[:, None, :, None])
    v8 = oracle.f32_to_e4m3(oracle.bf16_to_f64(vb).astype(np.float32) / vs[:, None, :, None])
    return pb, k8, v8, ks, vs


def _prefill_fp8_args(pb):
    return (pb.qo_indptr.numpy(), pb.kv_indptr.numpy(), pb.kv.req_to_token.numpy(),
            pb.kv.req_pool_indices.numpy(), pb.scale)


@pytest.mark.parametrize("Hq,Hkv,D,page", [(6, 3, 8, 4), (8, 2, 16, 1), (4, 4, 32, 16)])
def test_prefill_fp8_matches_masked_library_attention_on_dequantised_cache(Hq, Hkv, D, page):
    new, pre = [5, 17, 1, 9], [11, 0, 6, 32]
    pb, k8, v8, ks, vs = _fp8_prefill(new, pre, Hq, Hkv, D, page, seed=61 + D)
    out = oracle.prefill_fp8(bits(pb.q), k8, v8, pb.layer, *_prefill_fp8_args(pb), ks, vs)
    kf = _torch_e4m3_values(k8) * ks[:, None, :, None].astype(np.float64)
    vf = _torch_e4m3_values(v8) * vs[:, None, :, None].astype(np.float64)
    qf = oracle.bf16_to_f64(bits(pb.q))
    G = Hq // Hkv
    t0 = 0
    for r, (n, p) in enumerate(zip(new, pre)):
        row = int(pb.kv.req_pool_indices[r])
        slots = pb.kv.req_to_token[row, :p + n].numpy()
        mask = np.arange(p + n)[None, :] <= (p + np.arange(n))[:, None]   # bottom-right aligned
        for hq in range(Hq):
            ref = _sdpa_f64(qf[t0:t0 + n, hq], kf[pb.layer, slots, hq // G], vf[pb.layer, slots, hq // G],
                            pb.scale, mask=mask)
            np.testing.assert_allclose(out[t0:t0 + n, hq], ref, rtol=1e-12, atol=1e-12)
        t0 += n


def test_prefill_fp8_with_power_of_two_scales_equals_bf16_prefill():
    # e4m3 values times 2^k are bf16 numbers: the bf16 oracle on that cache
    # computes the same attention in the same order
    ks = np.array([[2.0 ** -5, 2.0 ** -7]], np.float32)
    vs = np.array([[2.0 ** -3, 1.0]], np.float32)
    pb, k8, v8, _, _ = _fp8_prefill([7, 3, 12], [4, 20, 0], 8, 2, 16, 4, seed=63, ks=ks, vs=vs)
    kbf = oracle.f64_to_bf16(oracle.e4m3_to_f64(k8) * ks[:, None, :, None])
    vbf = oracle.f64_to_bf16(oracle.e4m3_to_f64(v8) * vs[:, None, :, None])
    ref = oracle.prefill(bits(pb.q), kbf, vbf, pb.layer, *_prefill_fp8_args(pb))
    out = oracle.prefill_fp8(bits(pb.q), k8, v8, pb.layer, *_prefill_fp8_args(pb), ks, vs)
    np.testing.assert_array_equal(out, ref)


def test_prefill_fp8_last_row_equals_fp8_decode_and_selection_matches():
    new, pre = [7, 3, 12], [4, 20, 0]
    pb, k8, v8, ks, vs = _fp8_prefill(new, pre, 4, 1, 8, 4, seed=64)
    out = oracle.prefill_fp8(bits(pb.q), k8, v8, pb.layer, *_prefill_fp8_args(pb), ks, vs)
    last = pb.qo_indptr.numpy()[1:] - 1
    dec = oracle.decode_fp8(bits(pb.q)[last], k8, v8, pb.layer, pb.kv.req_to_token.numpy(),
                            pb.kv.req_pool_indices.numpy(), np.array([p + n for p, n in zip(pre, new)], np.int32),
                            pb.scale, ks, vs)
    np.testing.assert_array_equal(out[last], dec)
    sel = oracle.prefill_fp8(bits(pb.q), k8, v8, pb.layer, *_prefill_fp8_args(pb), ks, vs,
                             sel=(np.array([21, 0, 9], np.int32), np.array([3, 0, 2], np.int32)))
    np.testing.assert_array_equal(sel, out[[21, 0, 9], [3, 0, 2]])
