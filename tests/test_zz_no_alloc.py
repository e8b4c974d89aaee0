"""The allocation-free decode entry point against the workspace one and the oracle.

pa_paged_decode_attn_noalloc exists for callers that cannot allocate device
memory where decode runs -- for example a plugin whose host program owns every
device allocation, or a serving loop that must never call cudaMalloc because
it synchronises the device.  Instead of a caller workspace it uses a fixed
scratch array inside the library, shared by every call on the device.

This file is collected last so that a stop-at-first-failure run has already
run everything else; it also passes on its own in a fresh process.
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


def _step(seed, lens):
    """A decode step whose new K/V the library stores on the device; the
    expected cache is built on the host by the oracle's store from the same
    inputs."""
    st = W.make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=2, size=32768,
                            page_size=16, seed=seed, layer=1, max_ctx=4096, device="cuda")
    kb0, vb0 = bits(st.kv.k_buf), bits(st.kv.v_buf)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, st.k_new, st.v_new, st.loc)
    kb, vb = oracle.kv_store(kb0, vb0, st.layer, bits(st.k_new), bits(st.v_new), npy(st.loc))
    return st, kb, vb


def test_noalloc_matches_workspace_entry_point_twice():
    # Two calls in a row with different batches and lengths: the second call
    # must not see the first call's partials or merge tickets.  The first
    # batch has requests long enough to be split, so the merge path runs.
    # Same max_splits -> same split plan: the outputs must be identical.
    for seed, lens in ((11, [4000, 17, 900]), (12, [1, 2500, 64, 3000, 5, 1024])):
        st, kb, vb = _step(seed, lens)
        B, Hq, D = st.q.shape
        ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, 8, D, MAX_SPLITS))
        ref = torch.full_like(st.q, float("nan"))
        api.pa_paged_decode_attn(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                 st.kv.req_pool_indices, st.kv.seq_lens, st.scale, ws, MAX_SPLITS, ref)
        got = torch.full_like(st.q, float("nan"))
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        api.pa_paged_decode_attn_noalloc(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                         st.kv.req_pool_indices, st.kv.seq_lens, st.scale, MAX_SPLITS, got,
                                         error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert api.pa_get_error(ws) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"seed {seed}: not bit-identical"
        want = oracle.decode(bits(st.q), kb, vb, st.layer, npy(st.kv.req_to_token), npy(st.kv.req_pool_indices),
                             npy(st.kv.seq_lens), st.scale)
        assert_attention_close(npy(got.float()), want, f"no-alloc decode vs oracle, seed {seed}")
    # the error word is optional: the same call without it gives the same bits
    again = torch.full_like(st.q, float("nan"))
    api.pa_paged_decode_attn_noalloc(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                     st.kv.req_pool_indices, st.kv.seq_lens, st.scale, MAX_SPLITS, again)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), got.view(torch.int16))


def test_noalloc_rejects_batches_beyond_its_array():
    st, _, _ = _step(13, [64] * 20)   # 20 requests x 64 splits x 32 heads x 130 floats > 16 MiB
    out = torch.empty_like(st.q)
    with pytest.raises(api.PaError) as e:
        api.pa_paged_decode_attn_noalloc(st.q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token,
                                         st.kv.req_pool_indices, st.kv.seq_lens, st.scale, MAX_SPLITS, out)
    assert e.value.status == 5   # PA_ERR_WORKSPACE


def test_noalloc_failed_call_writes_nothing():
    # a call that fails validation copies no error word (the copy would
    # overwrite the -1) and leaves the output alone
    st, _, _ = _step(14, [300, 40])
    out = torch.full_like(st.q, 3.0)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(api.PaError) as e:
        api.pa_paged_decode_attn_noalloc(st.q, st.kv.k_buf, st.kv.v_buf, 2, st.kv.req_to_token,
                                         st.kv.req_pool_indices, st.kv.seq_lens, st.scale, MAX_SPLITS, out,
                                         error_word=err)   # layer 2 of a 2-layer cache
    assert e.value.status == 2   # PA_ERR_SHAPE
    torch.cuda.synchronize()
    assert int(err.item()) == -1
    assert (out == 3.0).all()
