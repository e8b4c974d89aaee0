"""Launch overlap (programmatic dependent launch) changes when kernels start,
never what they compute: chains in which each call reads what the previous
call wrote -- RoPE -> KV store -> decode, RoPE -> KV store -> prefill, and
back-to-back decodes sharing one workspace -- give bit-identical results with
overlap off, safe, early-metadata and early-KV, eagerly and under repeated graph
replay.  Early-KV mode copies cache rows other than each request's newest
one before the wait, which these chains allow (the store writes only the
newest rows)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_188_gb300 import api
from paged_kv_cache_188_gb300 import workloads as W

pytestmark = pytest.mark.gpu
MODES = [api.OVERLAP_OFF, api.OVERLAP_SAFE, api.OVERLAP_EARLY_METADATA, api.OVERLAP_EARLY_KV]


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()
    yield
    api.pa_set_launch_overlap(api.OVERLAP_OFF)


def _bits(t):
    return t.view(torch.int16).clone()


def _decode_chain(st, q0, k0, ws, outs, stream):
    """RoPE on fresh copies of q / k_new, store k/v, then decode on two layers."""
    q, k = st.q, st.k_new
    q.copy_(q0)
    k.copy_(k0)
    api.pa_rope_packed(q, k, st.positions, st.cos_tab, st.sin_tab, stream=stream)
    api.pa_kv_store(st.kv.k_buf, st.kv.v_buf, st.layer, k, st.v_new, st.loc, stream=stream)
    for out in outs:
        api.pa_paged_decode_attn(q, st.kv.k_buf, st.kv.v_buf, st.layer, st.kv.req_to_token, st.kv.req_pool_indices,
                                 st.kv.seq_lens, st.scale, ws, 64, out, stream=stream)


# 24 requests x 8 kv heads: more pairs than half the CTAs, so each decode
# call is the decode kernel and the deferred-merge kernel
LARGE = [int(x) for x in np.random.default_rng(24).integers(1, 4000, size=24)]


def _decode_state(lens=(3000, 17, 1200, 640)):
    st = W.make_decode_step(lens=list(lens), n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=2,
                            size=131072, page_size=16, seed=31, layer=1, max_ctx=4096, device="cuda")
    return st, st.q.clone(), st.k_new.clone()


@pytest.mark.parametrize("lens", [(3000, 17, 1200, 640), tuple(LARGE)], ids=["small", "large"])
def test_decode_chain_identical_across_modes_eager_and_graph(lens):
    st, q0, k0 = _decode_state(lens)
    B, Hq, D = st.q.shape
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, 8, D, 64))
    ref = None
    for mode in MODES:
        api.pa_set_launch_overlap(mode)
        outs = [torch.full_like(st.q, float("nan")) for _ in range(3)]
        _decode_chain(st, q0, k0, ws, outs, torch.cuda.current_stream())
        torch.cuda.synchronize()
        got = [_bits(o) for o in outs]
        if ref is None:
            ref = got
            assert torch.equal(got[0], got[1]) and torch.equal(got[0], got[2])
        for g, r in zip(got, ref):
            assert torch.equal(g, r), f"eager, mode {mode}"
        # the same chain captured once and replayed several times
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        gouts = [torch.zeros_like(st.q) for _ in range(3)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            _decode_chain(st, q0, k0, ws, gouts, s)
        for _ in range(4):
            for o in gouts:
                o.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            for o, r in zip(gouts, ref):
                assert torch.equal(_bits(o), r), f"graph, mode {mode}"
        assert api.pa_get_error(ws) == 0


def test_prefill_chain_identical_across_modes():
    pb = W.make_prefill_batch(new_lens=[300, 77, 1000], prefix_lens=[500, 0, 64], n_q_heads=32, n_kv_heads=8,
                              head_dim=128, size=8192, page_size=16, seed=32, device="cuda")
    q0, k0 = pb.q.clone(), pb.k_new.clone()
    ws = api.alloc_workspace(api.pa_prefill_workspace_bytes())
    ref = None
    for mode in MODES:
        api.pa_set_launch_overlap(mode)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        q, k = pb.q, pb.k_new
        outs = [torch.zeros_like(q) for _ in range(2)]

        def chain():
            q.copy_(q0)
            k.copy_(k0)
            api.pa_rope_packed(q, k, pb.positions, pb.cos_tab, pb.sin_tab, stream=s)
            api.pa_kv_store(pb.kv.k_buf, pb.kv.v_buf, 0, k, pb.v_new, pb.loc, stream=s)
            for o in outs:
                api.pa_paged_prefill_attn(q, pb.kv.k_buf, pb.kv.v_buf, 0, pb.qo_indptr, pb.kv_indptr,
                                          pb.kv.req_to_token, pb.kv.req_pool_indices, pb.scale, ws, o, stream=s)
        with torch.cuda.stream(s):
            chain()
        torch.cuda.synchronize()
        got = [_bits(o) for o in outs]
        if ref is None:
            ref = got
            assert torch.equal(got[0], got[1])
        for g_, r in zip(got, ref):
            assert torch.equal(g_, r), f"eager, mode {mode}"
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain()
        for _ in range(3):
            for o in outs:
                o.zero_()
            g.replay()
            torch.cuda.synchronize()
            for o, r in zip(outs, ref):
                assert torch.equal(_bits(o), r), f"graph, mode {mode}"
        words = ws.view(torch.int32)
        assert int(words[0]) == 0 and int(words[16]) == 0 and int(words[32]) == 0


def test_fused_steps_back_to_back_identical_across_modes():
    # two layers' fused steps sharing one workspace, eagerly and in a graph:
    # the second step's early index reads overlap the first step's tail
    st = W.make_decode_step(lens=[2000, 5, 900], n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=2,
                            size=8192, page_size=16, seed=41, layer=0, max_ctx=4096, fill_layers=[0, 1],
                            device="cuda")
    B, Hq, D = st.q.shape
    ws = api.alloc_workspace(api.pa_decode_workspace_bytes(B, Hq, 8, D, 64))
    kb0, vb0 = st.kv.k_buf.clone(), st.kv.v_buf.clone()
    ref = None
    for mode in MODES:
        api.pa_set_launch_overlap(mode)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        outs = [torch.zeros_like(st.q) for _ in range(2)]

        def steps():
            for layer, o in enumerate(outs):
                api.pa_decode_step(st.q, st.k_new, st.v_new, st.positions, st.cos_tab, st.sin_tab, st.kv.k_buf,
                                   st.kv.v_buf, layer, st.loc, st.kv.req_to_token, st.kv.req_pool_indices,
                                   st.kv.seq_lens, st.scale, ws, 64, o, stream=s)
        st.kv.k_buf.copy_(kb0)
        st.kv.v_buf.copy_(vb0)
        with torch.cuda.stream(s):
            steps()
        torch.cuda.synchronize()
        got = [_bits(o) for o in outs] + [_bits(st.kv.k_buf), _bits(st.kv.v_buf)]
        if ref is None:
            ref = got
        for g_, r in zip(got, ref):
            assert torch.equal(g_, r), f"eager, mode {mode}"
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            steps()
        for _ in range(3):
            for o in outs:
                o.zero_()
            g.replay()
            torch.cuda.synchronize()
            for o, r in zip(outs, ref):
                assert torch.equal(_bits(o), r), f"graph, mode {mode}"
        assert api.pa_get_error(ws) == 0
