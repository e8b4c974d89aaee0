"""Cascade (shared-prefix) decode against the float64 oracle and against
plain decode: groups whose page-table rows share their first tokens read the
shared prefix once per chunk of members; the result must stay within the
attention tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref| of the oracle."""
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


def _case(lens, hq, hkv, group_size, prefix, seed, d=128, size=65536):
    """The step's inputs, its new K/V stored on the device by the library, and
    the expected cache built on the host by the oracle's store from the same
    inputs (the oracle never sees a value the library wrote)."""
    st = W.make_decode_step(lens=lens, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, n_layers=1, size=size,
                            page_size=16, seed=seed, max_ctx=max(lens) + 16, shared_prefix=(group_size, prefix),
                            device="cuda")
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    kb, vb = oracle.kv_store(kb0, vb0, st.layer, bits(st.k_new), bits(st.v_new), npy(st.loc))
    return st, kb, vb


def _ref(st, kb, vb):
    return oracle.decode(bits(st.q), kb, vb, st.layer, npy(st.kv.req_to_token),
                         npy(st.kv.req_pool_indices), npy(st.kv.seq_lens), st.scale)


def _cascade(st, indptr, reqs, prefix, caps):
    B, Hq, D = st.q.shape
    ws = api.alloc_workspace(api.pa_cascade_workspace_bytes(*caps, Hq, st.kv.k_buf.shape[2], D))
    out = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn_cascade(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                     st.kv.req_pool_indices, st.kv.seq_lens, indptr.cuda(), reqs.cuda(),
                                     prefix.cuda(), st.scale, ws, caps, out)
    torch.cuda.synchronize()
    return out, ws


@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (32, 2), (8, 8)])
def test_cascade_matches_oracle(hq, hkv):
    # groups of 5 (chunks of 16/G members leave partial chunks), ragged lengths,
    # one member shorter than the prefix window
    lens = [3000, 1500, 700, 2500, 130, 4000, 1100, 900, 2048, 5000, 64]
    st, kb, vb = _case(lens, hq, hkv, 5, 512, seed=hq + hkv)
    indptr, reqs, prefix = W.prefix_groups(lens, 5, 512, 16)
    caps = (len(lens), 3, 5, MAX_SPLITS)
    out, ws = _cascade(st, indptr, reqs, prefix, caps)
    assert api.pa_get_error(ws) == 0
    assert_attention_close(npy(out.float()), _ref(st, kb, vb), f"cascade hq={hq} hkv={hkv}")


def test_cascade_config3_shape_and_repeat_calls():
    lens = W.cfg_lens_uniform(32, 512, 8192, seed=3)
    st, kb, vb = _case(lens, 32, 8, 8, 1024, seed=3, size=262144)
    indptr, reqs, prefix = W.prefix_groups(lens, 8, 1024, 16)
    caps = (32, 4, 8, MAX_SPLITS)
    out, ws = _cascade(st, indptr, reqs, prefix, caps)
    ref = _ref(st, kb, vb)
    assert_attention_close(npy(out.float()), ref, "cascade config-3 shape")
    # a second call on the same workspace (tickets back at zero), then groups
    # that leave requests out: the results stay within tolerance
    B, Hq, D = st.q.shape
    out2 = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn_cascade(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                     st.kv.req_pool_indices, st.kv.seq_lens, indptr.cuda(), reqs.cuda(),
                                     prefix.cuda(), st.scale, ws, caps, out2)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    sub_indptr = torch.tensor([0, 3, 3, 5], dtype=torch.int32)            # group 1 empty
    sub_reqs = torch.tensor([0, 1, 2, 8, 9], dtype=torch.int32)
    sub_prefix = torch.tensor([int(prefix[0]), 0, int(prefix[1])], dtype=torch.int32)
    out3 = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn_cascade(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                     st.kv.req_pool_indices, st.kv.seq_lens, sub_indptr.cuda(), sub_reqs.cuda(),
                                     sub_prefix.cuda(), st.scale, ws, caps, out3)
    torch.cuda.synchronize()
    assert api.pa_get_error(ws) == 0
    assert_attention_close(npy(out3.float()), ref, "cascade with partial groups")
    # no groups: plain decode through the same workspace
    out4 = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn_cascade(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                     st.kv.req_pool_indices, st.kv.seq_lens, torch.zeros(1, dtype=torch.int32).cuda(),
                                     torch.zeros(1, dtype=torch.int32).cuda(), torch.zeros(0, dtype=torch.int32).cuda(),
                                     st.scale, ws, caps, out4)
    torch.cuda.synchronize()
    assert_attention_close(npy(out4.float()), ref, "cascade without groups")
