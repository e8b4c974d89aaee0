"""Test plumbing: moving inputs between the device and the oracle, and the
tolerances the parity tests use.  No attention arithmetic lives here."""
import numpy as np
import torch

# attention outputs: |gpu - ref| <= ATOL + RTOL * |ref| (bf16 inputs, fp32 accumulation)
ATOL = 1e-2
RTOL = 1e-2


def bits(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def npy(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_attention_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    worst = float(excess.max()) if excess.size else -1.0
    if worst > 0:
        i = np.unravel_index(int(np.argmax(excess)), excess.shape)
        raise AssertionError(f"{what}: |gpu-ref| exceeds {ATOL}+{RTOL}|ref| by {worst:.3e} at {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r}")


def bf16_ulp_distance(a_bits, b_bits) -> np.ndarray:
    """Distance in units in the last place between two bf16 bit-pattern arrays."""
    def key(x):
        x = x.astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(key(np.asarray(a_bits)) - key(np.asarray(b_bits)))


def compact_requests(k_buf, v_buf, layer, req_to_token, req_pool_indices, seq_lens, reqs):
    """Host copies of just the cache rows that requests ``reqs`` address.

    Returns (k [1, U, Hkv, D] bits, v bits, r2t [len(reqs), max_n] int32,
    rows [len(reqs)] = arange, lens).  Slots are renumbered 0..U-1 in sorted
    order; by the oracle's page-placement invariance the attention result is
    unchanged."""
    reqs = list(reqs)
    rows = req_pool_indices[reqs].long()
    lens = seq_lens[reqs].long()
    max_n = max(1, int(lens.max()))
    parts = [req_to_token[int(r), :int(n)].long() for r, n in zip(rows.tolist(), lens.tolist())]
    allslots = torch.cat(parts) if parts else torch.zeros(0, dtype=torch.long, device=req_to_token.device)
    uniq, inv = torch.unique(allslots, return_inverse=True)
    k = bits(k_buf[layer, uniq])[None]
    v = bits(v_buf[layer, uniq])[None]
    r2t = np.full((len(reqs), max_n), -1, np.int32)
    inv = npy(inv)
    off = 0
    for i, n in enumerate(lens.tolist()):
        r2t[i, :n] = inv[off:off + n]
        off += n
    return k, v, r2t, np.arange(len(reqs), dtype=np.int32), npy(lens).astype(np.int32)
