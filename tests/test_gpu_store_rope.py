"""GPU parity of the KV store (bit-exact) and packed RoPE (<= 1 bf16 ulp)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W
from _helpers import bf16_ulp_distance, bits, npy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


@pytest.mark.parametrize("T,Hkv,D", [(1, 2, 64), (37, 8, 128), (1000, 1, 64), (513, 4, 8)])
def test_kv_store_bit_exact_whole_buffer(T, Hkv, D):
    g = W.generator(T + D)
    kb = W.nan_filled((3, 4096, Hkv, D)).cuda()
    vb = W.nan_filled((3, 4096, Hkv, D)).cuda()
    kb[0, :100] = W.bf16_normal((100, Hkv, D), g).cuda()
    kn = W.bf16_normal((T, Hkv, D), g)
    vn = W.bf16_normal((T, Hkv, D), g)
    loc = torch.randperm(4096, generator=g)[:T].to(torch.int32)
    kw, vw = oracle.kv_store(bits(kb), bits(vb), 2, bits(kn), bits(vn), npy(loc))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_kv_store(kb, vb, 2, kn.cuda(), vn.cuda(), loc.cuda(), error_word=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(kb), kw)
    np.testing.assert_array_equal(bits(vb), vw)
    assert int(err) == 0


def test_kv_store_bad_location_skipped_and_flagged():
    kb = W.nan_filled((1, 64, 2, 8)).cuda()
    vb = W.nan_filled((1, 64, 2, 8)).cuda()
    before_k, before_v = bits(kb), bits(vb)
    g = W.generator(3)
    kn, vn = W.bf16_normal((3, 2, 8), g), W.bf16_normal((3, 2, 8), g)
    loc = torch.tensor([5, 64, -1], dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_kv_store(kb, vb, 0, kn.cuda(), vn.cuda(), loc.cuda(), error_word=err)
    assert api.pa_get_error_word(err) & api.DEVERR_SLOT
    kw, vw = oracle.kv_store(before_k, before_v, 0, bits(kn)[:1], bits(vn)[:1], npy(loc)[:1])
    np.testing.assert_array_equal(bits(kb), kw)
    np.testing.assert_array_equal(bits(vb), vw)


def test_kv_store_config4_full_size():
    """Packed-prefill store: ~17K new tokens into random free slots of a [1, 65536, 8, 128] cache."""
    pb = W.config4(device="cuda")
    kb0, vb0 = bits(pb.kv.k_buf), bits(pb.kv.v_buf)
    api.pa_kv_store(pb.kv.k_buf, pb.kv.v_buf, 0, pb.k_new, pb.v_new, pb.loc)
    torch.cuda.synchronize()
    kw, vw = oracle.kv_store(kb0, vb0, 0, bits(pb.k_new), bits(pb.v_new), npy(pb.loc))
    np.testing.assert_array_equal(bits(pb.kv.k_buf), kw)
    np.testing.assert_array_equal(bits(pb.kv.v_buf), vw)


def test_kv_store_config5_full_size_properties():
    """256 tokens into a [1, 16M, 8, 128] cache: written rows equal the inputs
    bit for bit, and no other byte of either buffer changes."""
    st = W.config5(device="cuda")
    before_k = st.kv.k_buf.view(torch.int16).clone()
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, 0, st.k_new, st.v_new, st.loc)
    torch.cuda.synchronize()
    loc = st.loc.long()
    assert torch.equal(st.kv.k_buf[0, loc].view(torch.int16), st.k_new.view(torch.int16))
    assert torch.equal(st.kv.v_buf[0, loc].view(torch.int16), st.v_new.view(torch.int16))
    after_k = st.kv.k_buf.view(torch.int16)
    after_k_rows = after_k[0, loc].clone()
    after_k[0, loc] = before_k[0, loc]
    assert torch.equal(after_k, before_k)
    after_k[0, loc] = after_k_rows


@pytest.mark.parametrize("T,Hq,Hkv,D", [(1, 8, 2, 64), (256, 64, 8, 128), (333, 32, 8, 128), (5, 3, 0, 16)])
def test_rope_within_one_ulp(T, Hq, Hkv, D):
    g = W.generator(T * 3 + Hq)
    q = W.bf16_normal((T, Hq, D), g)
    k = W.bf16_normal((T, Hkv, D), g) if Hkv else None
    cos, sin = W.rope_tables(W.ROPE_MAX_POS, D)
    pos = torch.randint(0, W.ROPE_MAX_POS, (T,), generator=g, dtype=torch.int32)
    pos[0] = 0
    pos[-1] = W.ROPE_MAX_POS - 1
    qd = q.cuda()
    kd = k.cuda() if k is not None else None
    api.pa_rope_packed(qd, kd, pos.cuda(), cos.cuda(), sin.cuda())
    torch.cuda.synchronize()
    qr, _ = oracle.rope(bits(q), npy(pos), npy(cos), npy(sin))
    assert bf16_ulp_distance(bits(qd), qr).max() <= 1
    if k is not None:
        kr, _ = oracle.rope(bits(k), npy(pos), npy(cos), npy(sin))
        assert bf16_ulp_distance(bits(kd), kr).max() <= 1
    if T > 1:   # position 0 is the identity, exactly
        np.testing.assert_array_equal(bits(qd)[0], bits(q)[0])


def test_rope_config4_full_size():
    pb = W.config4(device="cuda")
    q, k = pb.q.clone(), pb.k_new.clone()
    api.pa_rope_packed(q, k, pb.positions, pb.cos_tab, pb.sin_tab)
    torch.cuda.synchronize()
    pos, ct, sn = npy(pb.positions), npy(pb.cos_tab), npy(pb.sin_tab)
    qr, _ = oracle.rope(bits(pb.q), pos, ct, sn)
    kr, _ = oracle.rope(bits(pb.k_new), pos, ct, sn)
    assert bf16_ulp_distance(bits(q), qr).max() <= 1
    assert bf16_ulp_distance(bits(k), kr).max() <= 1


def test_rope_bad_position_flagged_and_untouched():
    g = W.generator(4)
    q = W.bf16_normal((3, 2, 64), g).cuda()
    q0 = q.clone()
    cos, sin = W.rope_tables(128, 64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.pa_rope_packed(q, None, torch.tensor([1, 128, 5], dtype=torch.int32, device="cuda"), cos.cuda(),
                       sin.cuda(), error_word=err)
    assert api.pa_get_error_word(err) & api.DEVERR_POS
    assert torch.equal(q[1].view(torch.int16), q0[1].view(torch.int16))
    assert not torch.equal(q[0].view(torch.int16), q0[0].view(torch.int16))
