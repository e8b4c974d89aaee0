"""Seeded synthetic inputs for the paged-KV attention path.

This module only draws inputs: random bf16 values, page assignments, request
rows, lengths and the rotary cos/sin table.  It holds none of the attention,
rotary or store arithmetic, so both the CUDA path and the float64 oracle can be
fed from it without sharing any of the computation.

Layout conventions (AstrAI commit 398e8a3, tests/inference/test_cache.py: per
layer [n_layers, size, n_kv_heads, head_dim] KV buffers addressed
buffer[layer_id, loc]; int32 page-table, request-row and location indices):

* ``k_buf``/``v_buf``: bf16 ``[n_layers, size, Hkv, D]``.  Slots no request
  uses hold the bf16 NaN pattern 0x7FC0 as a canary, so a stray read shows up.
* ``req_to_token``: int32 ``[req_rows, max_ctx]``; request ``b`` lives in row
  ``req_pool_indices[b]`` and its token ``j`` at slot ``req_to_token[row, j]``.
  Entries past a request's length hold stale garbage (old slots, negative and
  out-of-range values) that a correct reader never touches.
* Pages: slot ``page * page_size + j % page_size`` for logical token ``j`` on
  the request's ``j // page_size``-th page; pages come from one ``randperm``.

Values are N(0, 1) drawn in fp32 from a seeded ``torch.Generator`` and rounded
to bf16 (round to nearest even, torch's conversion).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16_NAN = 0x7FC0
ROPE_THETA = 10000.0
ROPE_MAX_POS = 32768


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def bf16_normal(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def nan_filled(shape, device="cpu") -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.int16, device=device)
    t.fill_(BF16_NAN)
    return t.view(torch.bfloat16)


def rope_tables(max_pos: int, head_dim: int, theta: float = ROPE_THETA):
    """cos/sin tables, fp32 ``[max_pos, head_dim // 2]``.

    Entry (p, i) is cos / sin of the angle p * theta^(-2i/D), evaluated in
    float64 (an fp32 product loses bits near p = 32K) and rounded once to fp32.
    """
    half = head_dim // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / head_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).to(torch.float32), torch.sin(ang).to(torch.float32)


@dataclass
class PagedKV:
    """A filled paged cache plus the request table that addresses it."""
    k_buf: torch.Tensor           # bf16 [n_layers, size, Hkv, D]
    v_buf: torch.Tensor
    req_to_token: torch.Tensor    # int32 [req_rows, max_ctx]
    req_pool_indices: torch.Tensor  # int32 [B]
    seq_lens: torch.Tensor        # int32 [B] (tokens whose K/V are addressed)
    page_size: int
    used_slots: torch.Tensor = field(repr=False, default=None)  # int64, unique slots in use


def _assign_slots(lens, page_size, n_pages, gen, shared_prefix=None):
    """Per request, the slot of every logical token, page-granular.

    ``shared_prefix``: optional (group_size, prefix_len); requests of one group
    map their first tokens, up to prefix_len, onto the group's common pages
    (radix-style prefix reuse), the rest onto private pages.  The page that
    holds a request's last token is always private."""
    perm = torch.randperm(n_pages, generator=gen)
    nxt = 0

    def take(k):
        nonlocal nxt
        if nxt + k > n_pages:
            raise ValueError("cache too small for the requested lengths")
        p = perm[nxt:nxt + k]
        nxt += k
        return p

    slots_per_req = []
    group_pages = {}
    for b, n in enumerate(lens):
        n = int(n)
        n_req_pages = -(-n // page_size)
        if shared_prefix is not None:
            gsz, plen = shared_prefix
            assert plen % page_size == 0
            g = b // gsz
            if g not in group_pages:
                group_pages[g] = take(plen // page_size)
            # the page holding the request's newest token stays private: a
            # request never writes into pages it shares with others
            k_shared = min(max(n - 1, 0) // page_size, plen // page_size)
            pages = torch.cat([group_pages[g][:k_shared], take(n_req_pages - k_shared)])
        else:
            pages = take(n_req_pages)
        j = torch.arange(n, dtype=torch.int64)
        slots_per_req.append(pages[j // page_size] * page_size + j % page_size)
    return slots_per_req


def make_paged_kv(*, lens, n_layers, size, n_kv_heads, head_dim, page_size, seed,
                  max_ctx=None, req_rows=None, shared_prefix=None, device="cpu",
                  fill_layers=None, unfilled_tail=0) -> PagedKV:
    """Build buffers and tables for ``len(lens)`` requests.

    ``fill_layers``: layers whose used slots receive random values (default
    all).  ``unfilled_tail``: the last ``unfilled_tail`` tokens of each request
    keep the NaN canary (their K/V are written later by the store under test).
    """
    gen = generator(seed)
    B = len(lens)
    lens = [int(x) for x in lens]
    max_ctx = max_ctx or max(max(lens, default=1), 1)
    req_rows = req_rows or max(B, 1)
    assert size % page_size == 0
    slots = _assign_slots(lens, page_size, size // page_size, gen, shared_prefix)

    # request rows: a random injective map, the other rows hold garbage
    rows = torch.randperm(req_rows, generator=gen)[:B].to(torch.int32)
    stale = torch.randint(-size, 2 * size, (req_rows, max_ctx), generator=gen, dtype=torch.int64)
    r2t = stale.to(torch.int32)
    for b in range(B):
        r2t[rows[b], :lens[b]] = slots[b].to(torch.int32)

    k_buf = nan_filled((n_layers, size, n_kv_heads, head_dim), device)
    v_buf = nan_filled((n_layers, size, n_kv_heads, head_dim), device)
    keep = [s[: max(len(s) - unfilled_tail, 0)] for s in slots]
    used = torch.unique(torch.cat(keep)) if keep else torch.zeros(0, dtype=torch.int64)
    layers = range(n_layers) if fill_layers is None else fill_layers
    vgen = generator(seed + 7919, device)
    used_dev = used.to(device)
    chunk = max(1, (1 << 26) // max(1, n_kv_heads * head_dim))
    for layer in layers:
        for c0 in range(0, used.numel(), chunk):
            idx = used_dev[c0:c0 + chunk]
            k_buf[layer, idx] = bf16_normal((idx.numel(), n_kv_heads, head_dim), vgen, device)
            v_buf[layer, idx] = bf16_normal((idx.numel(), n_kv_heads, head_dim), vgen, device)
    return PagedKV(k_buf, v_buf, r2t.to(device), rows.to(device),
                   torch.tensor(lens, dtype=torch.int32, device=device), page_size, used)


@dataclass
class DecodeStep:
    """One decode step: the new token of every request plus the cache."""
    kv: PagedKV
    q: torch.Tensor          # bf16 [B, Hq, D] (before rotary)
    k_new: torch.Tensor      # bf16 [B, Hkv, D] (before rotary)
    v_new: torch.Tensor      # bf16 [B, Hkv, D]
    positions: torch.Tensor  # int32 [B] = seq_lens - 1
    loc: torch.Tensor        # int32 [B]: slot of the new token
    cos_tab: torch.Tensor
    sin_tab: torch.Tensor
    scale: float
    layer: int


def make_decode_step(*, lens, n_q_heads, n_kv_heads, head_dim, n_layers, size, page_size,
                     seed, layer=0, max_ctx=None, req_rows=None, shared_prefix=None,
                     device="cpu", fill_layers=None, max_pos=ROPE_MAX_POS) -> DecodeStep:
    """Cache holding every request's first seq_len-1 tokens; the step's new
    token (position seq_len-1) is stored by the step itself."""
    kv = make_paged_kv(lens=lens, n_layers=n_layers, size=size, n_kv_heads=n_kv_heads,
                       head_dim=head_dim, page_size=page_size, seed=seed, max_ctx=max_ctx,
                       req_rows=req_rows, shared_prefix=shared_prefix, device=device,
                       fill_layers=fill_layers, unfilled_tail=1)
    gen = generator(seed + 104729, device)
    B = len(lens)
    q = bf16_normal((B, n_q_heads, head_dim), gen, device)
    k_new = bf16_normal((B, n_kv_heads, head_dim), gen, device)
    v_new = bf16_normal((B, n_kv_heads, head_dim), gen, device)
    lens_t = kv.seq_lens.to(torch.int64)
    positions = (lens_t - 1).clamp(min=0).to(torch.int32)
    rows = kv.req_pool_indices.to(torch.int64)
    loc = kv.req_to_token[rows, positions.to(torch.int64)].to(torch.int32)
    cos_t, sin_t = rope_tables(max_pos, head_dim)
    return DecodeStep(kv, q, k_new, v_new, positions, loc, cos_t.to(device), sin_t.to(device),
                      1.0 / math.sqrt(head_dim), layer)


@dataclass
class PrefillBatch:
    """Packed prompts: new tokens of R requests after their cached prefixes."""
    kv: PagedKV              # seq_lens = total length L_r = prefix + new
    q: torch.Tensor          # bf16 [T, Hq, D] (before rotary)
    k_new: torch.Tensor      # bf16 [T, Hkv, D] (before rotary)
    v_new: torch.Tensor      # bf16 [T, Hkv, D]
    qo_indptr: torch.Tensor  # int32 [R+1]
    kv_indptr: torch.Tensor  # int32 [R+1]
    positions: torch.Tensor  # int32 [T]: prefix_len + i
    loc: torch.Tensor        # int32 [T]: slot of each new token
    prefix_lens: list
    new_lens: list
    cos_tab: torch.Tensor
    sin_tab: torch.Tensor
    scale: float
    layer: int


def make_prefill_batch(*, new_lens, prefix_lens, n_q_heads, n_kv_heads, head_dim, size,
                       page_size, seed, n_layers=1, layer=0, req_rows=None, max_ctx=None,
                       device="cpu", max_pos=ROPE_MAX_POS) -> PrefillBatch:
    new_lens = [int(x) for x in new_lens]
    prefix_lens = [int(x) for x in prefix_lens]
    R = len(new_lens)
    totals = [p + n for p, n in zip(prefix_lens, new_lens)]
    # build the cache with only the prefixes filled: the new tokens' slots keep
    # the canary until the store under test writes them
    kv = make_paged_kv(lens=totals, n_layers=n_layers, size=size, n_kv_heads=n_kv_heads,
                       head_dim=head_dim, page_size=page_size, seed=seed, max_ctx=max_ctx,
                       req_rows=req_rows, device="cpu", fill_layers=[])
    gen = generator(seed + 7919)
    for b in range(R):
        row = int(kv.req_pool_indices[b])
        pre = kv.req_to_token[row, :prefix_lens[b]].to(torch.int64)
        kv.k_buf[layer, pre] = bf16_normal((pre.numel(), n_kv_heads, head_dim), gen)
        kv.v_buf[layer, pre] = bf16_normal((pre.numel(), n_kv_heads, head_dim), gen)
    T = sum(new_lens)
    qo = torch.zeros(R + 1, dtype=torch.int32)
    kvp = torch.zeros(R + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(torch.tensor(new_lens, dtype=torch.int64), 0).to(torch.int32)
    kvp[1:] = torch.cumsum(torch.tensor(totals, dtype=torch.int64), 0).to(torch.int32)
    pos = torch.cat([torch.arange(p, p + n, dtype=torch.int32) for p, n in zip(prefix_lens, new_lens)]) \
        if T else torch.zeros(0, dtype=torch.int32)
    loc = torch.cat([kv.req_to_token[int(kv.req_pool_indices[b]), prefix_lens[b]:totals[b]]
                     for b in range(R)]) if T else torch.zeros(0, dtype=torch.int32)
    qgen = generator(seed + 104729)
    q = bf16_normal((T, n_q_heads, head_dim), qgen)
    k_new = bf16_normal((T, n_kv_heads, head_dim), qgen)
    v_new = bf16_normal((T, n_kv_heads, head_dim), qgen)
    cos_t, sin_t = rope_tables(max_pos, head_dim)
    kv = PagedKV(kv.k_buf.to(device), kv.v_buf.to(device), kv.req_to_token.to(device),
                 kv.req_pool_indices.to(device), kv.seq_lens.to(device), page_size, kv.used_slots)
    return PrefillBatch(kv, q.to(device), k_new.to(device), v_new.to(device), qo.to(device),
                        kvp.to(device), pos.to(device), loc.to(torch.int32).to(device),
                        prefix_lens, new_lens, cos_t.to(device), sin_t.to(device),
                        1.0 / math.sqrt(head_dim), layer)


# ---------------------------------------------------------------- configs
# The five workloads the path is exercised on.  Lengths are drawn here, once,
# from their seeds.

def cfg_lens_uniform(n, lo, hi, seed):
    g = generator(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def cfg_lens_lognormal(n, median, sigma, cap, seed):
    g = generator(seed)
    z = torch.randn(n, generator=g, dtype=torch.float64)
    return [int(min(cap, max(1, round(math.exp(math.log(median) + sigma * float(v)))))) for v in z]


def prefix_groups(lens, group_size, prefix_len, page_size):
    """Group arrays of a batch built with ``shared_prefix=(group_size, prefix_len)``:
    members of group g are requests g*group_size .. ; the common prefix is the
    shortest shared part of its members (the page holding a request's newest
    token is private).  Returns int32 tensors (indptr, reqs, prefix)."""
    B = len(lens)
    n_groups = -(-B // group_size)
    indptr = [min(g * group_size, B) for g in range(n_groups + 1)]
    reqs = list(range(B))
    prefix = []
    for g in range(n_groups):
        members = range(indptr[g], indptr[g + 1])
        prefix.append(min(min(max(int(lens[b]) - 1, 0) // page_size, prefix_len // page_size) * page_size
                          for b in members))
    return (torch.tensor(indptr, dtype=torch.int32), torch.tensor(reqs, dtype=torch.int32),
            torch.tensor(prefix, dtype=torch.int32))


def config1(device="cpu"):
    """Single-layer paged decode, B=1, Hq=8, Hkv=2, D=64, seq 256, 16 pages."""
    return make_decode_step(lens=[256], n_q_heads=8, n_kv_heads=2, head_dim=64, n_layers=1,
                            size=4096, page_size=16, seed=1, device=device)


def config2(seq_len, device="cpu", fill_layers=None):
    """B=1 decode, Hq=32, Hkv=8, D=128, 32 layers x 65536 slots, layer 17."""
    return make_decode_step(lens=[seq_len], n_q_heads=32, n_kv_heads=8, head_dim=128,
                            n_layers=32, size=65536, page_size=16, seed=2, layer=17,
                            max_ctx=32768, device=device, fill_layers=fill_layers)


def config3(device="cpu"):
    """B=32 ragged decode, seq U[512, 8192], 4 groups of 8 share 1024-token prefixes."""
    lens = cfg_lens_uniform(32, 512, 8192, seed=3)
    return make_decode_step(lens=lens, n_q_heads=32, n_kv_heads=8, head_dim=128, n_layers=1,
                            size=262144, page_size=16, seed=3, max_ctx=8192,
                            shared_prefix=(8, 1024), device=device)


def config4(device="cpu"):
    """16 packed prompts, new U[64, 2048], cached prefix U[0, 1024], Hq=32, Hkv=8."""
    new = cfg_lens_uniform(16, 64, 2048, seed=4)
    pre = cfg_lens_uniform(16, 0, 1024, seed=40)
    return make_prefill_batch(new_lens=new, prefix_lens=pre, n_q_heads=32, n_kv_heads=8,
                              head_dim=128, size=65536, page_size=16, seed=4, max_ctx=4096,
                              device=device)


def config5_lens():
    return cfg_lens_lognormal(256, 2048, 1.0, 32768, seed=5)


def config5(device="cpu"):
    """B=256, Hq=64, Hkv=8, token-granular pages over a 16M-slot buffer."""
    return make_decode_step(lens=config5_lens(), n_q_heads=64, n_kv_heads=8, head_dim=128,
                            n_layers=1, size=1 << 24, page_size=1, seed=5, max_ctx=32768,
                            device=device)
