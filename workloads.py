"""Seeded synthetic inputs for the KDA state path (shared by tests, smoke and bench).

This module only draws and packs inputs; it holds none of the method's
arithmetic (no gate or beta activation, no recurrence).  Both the CUDA library
and the CPU oracle consume what it returns: the oracle after an exact widening
of the stored values to float64.

Recipe (the serving pages print no dataset for this path, so every workload is
synthetic):
  * numpy Generator(PCG64(seed)); draw order: lengths / slots / plan integers,
    then q, k, v, raw beta, raw gate, then state pools.
  * q, k ~ N(0,1), L2-normalised per (token, head) over the key channels in fp32.
  * v ~ N(0,1); raw beta ~ N(0,1) (the kernels apply sigmoid);
    raw gate ~ N(0,1) per key channel (the kernels apply g = -softplus).
  * stored as bf16 (round-to-nearest-even) or kept fp32, per workload.
  * state pools ~ N(0, 0.1^2) fp32 (standard deviation 0.1).
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# bf16 storage helpers (representation only)


def f32_to_bf16_bits(x):
    """Round float32 to bf16 (nearest-even) and return the 16-bit patterns."""
    x = np.ascontiguousarray(x, np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    bias = ((b >> 16) & 1) + 0x7FFF
    out = ((b + bias) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits):
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def widen(a, dtype):
    """Stored representation -> float64 (exact)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, np.float32).astype(np.float64)


def store(x32, dtype):
    """float32 values -> stored representation for ``dtype`` ('bf16' or 'f32')."""
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    return np.ascontiguousarray(x32, np.float32)


# --------------------------------------------------------------------------
# activations of one batch of tokens


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def _l2norm(x):
    n = np.sqrt(np.sum(x.astype(np.float32) ** 2, axis=-1, keepdims=True, dtype=np.float32))
    return (x / np.maximum(n, np.float32(1e-30))).astype(np.float32)


def draw_tokens(rng, T, H, dk, dv, dtype):
    """q, k, v, raw beta, raw gate for T token rows, in the documented order."""
    q = _l2norm(_normal(rng, (T, H, dk)))
    k = _l2norm(_normal(rng, (T, H, dk)))
    v = _normal(rng, (T, H, dv))
    beta = _normal(rng, (T, H))
    gate = _normal(rng, (T, H, dk))
    return {k_: store(a, dtype) for k_, a in
            (("q", q), ("k", k), ("v", v), ("beta", beta), ("gate", gate))}


def draw_pool(rng, P, H, dv, dk, std=0.1):
    return (_normal(rng, (P, H, dv, dk)) * np.float32(std)).astype(np.float32)


# --------------------------------------------------------------------------
# workloads


def prefill_case(seed, lengths, H, *, dk=128, dv=128, dtype="bf16", chunk=64, pool_slots=0,
                 with_init=True, track_per_seq=1, track=None):
    """Packed varlen prefill.

    lengths: list of sequence lengths.  pool_slots > 0: a pool of that many
    slots; each sequence gets a distinct seeded slot used as init and final
    slot (in place).  track: explicit [N, M] chunk indices, else
    track_per_seq indices drawn uniformly in [0, n_chunks-1] (-1 for empty
    sequences)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = [int(x) for x in lengths]
    N = len(lengths)
    cu = np.zeros(N + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    slots = None
    if pool_slots:
        slots = rng.permutation(pool_slots)[:N].astype(np.int32)
    if track is None:
        track = np.full((N, track_per_seq), -1, np.int32)
        for n, L in enumerate(lengths):
            nc = (L + chunk - 1) // chunk
            if nc > 0:
                track[n] = rng.integers(0, nc, size=track_per_seq)
    track = np.asarray(track, np.int32).reshape(N, -1)
    tok = draw_tokens(rng, int(cu[-1]), H, dk, dv, dtype)
    pool = draw_pool(rng, pool_slots, H, dv, dk) if pool_slots else None
    init = slots if (slots is not None and with_init) else np.full(N, -1, np.int32)
    final = slots if slots is not None else np.full(N, -1, np.int32)
    return dict(tok, dtype=dtype, cu_seqlens=cu, N=N, T=int(cu[-1]), H=H, dk=dk, dv=dv,
                chunk=chunk, pool=pool, init_slot=init, final_slot=final, track=track,
                lengths=lengths)


def decode_case(seed, R, H, P, *, dk=128, dv=128, dtype="bf16", skip=()):
    """R requests, one token each, distinct seeded slots of a P-slot pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    slot = rng.permutation(P)[:R].astype(np.int32)
    for r in skip:
        slot[r] = -1
    tok = draw_tokens(rng, R, H, dk, dv, dtype)
    pool = draw_pool(rng, P, H, dv, dk)
    return dict(tok, dtype=dtype, R=R, H=H, dk=dk, dv=dv, pool=pool, slot=slot)


def spec_case(seed, R, K, H, *, P=None, dk=128, dv=128, dtype="bf16", q_len=None):
    """Speculative verify + commit: one checkpoint slot per request, K positions,
    accepted lengths uniform in {0..q_len}."""
    rng = np.random.Generator(np.random.PCG64(seed))
    P = R if P is None else P
    ckpt = rng.permutation(P)[:R].astype(np.int32)
    ql = np.full(R, K, np.int32) if q_len is None else np.asarray(q_len, np.int32)
    acc = np.array([rng.integers(0, int(x) + 1) for x in ql], np.int32)
    tok = draw_tokens(rng, R * K, H, dk, dv, dtype)
    pool = draw_pool(rng, P, H, dv, dk)
    return dict(tok, dtype=dtype, R=R, K=K, H=H, dk=dk, dv=dv, pool=pool, ckpt=ckpt,
                q_len=ql, num_accepted=acc)


def accept_case(seed, R, K, *, q_len=None, p_match=0.7, vocab=1 << 17):
    """Draft and sampled token ids for R speculative requests of up to K
    positions.  tokens[r, 0] is the last committed id, tokens[r, 1:] the drafts;
    sampled[r, i] repeats draft i+1 with probability p_match and is a fresh
    uniform id otherwise, so runs of agreement have a geometric length.
    Entries at or past q_len are junk ids that the acceptance must ignore."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ql = np.full(R, K, np.int32) if q_len is None else np.asarray(q_len, np.int32)
    tokens = rng.integers(0, vocab, size=(R, K), dtype=np.int64).astype(np.int32)
    fresh = rng.integers(0, vocab, size=(R, K), dtype=np.int64).astype(np.int32)
    keep = rng.random((R, K)) < p_match
    sampled = fresh.copy()
    sampled[:, :K - 1] = np.where(keep[:, :K - 1], tokens[:, 1:], fresh[:, :K - 1])
    return dict(tokens=tokens, sampled=sampled, q_len=ql, R=R, K=K)


def conv_case(seed, R, K, keep, channels, n_pools, P, *, dtype="bf16"):
    """Short-convolution pools for R speculative requests: n_pools tensors of
    [P, keep + K, channels] (the history rows, then room for K step inputs),
    values ~ N(0, 1) stored as bf16 or fp32, distinct seeded slots, and
    accepted lengths uniform in {0..K}."""
    rng = np.random.Generator(np.random.PCG64(seed))
    slots = rng.permutation(P)[:R].astype(np.int32)
    acc = rng.integers(0, K + 1, size=R).astype(np.int32)
    pools = []
    for _ in range(n_pools):
        x = rng.standard_normal((P, keep + K, channels)).astype(np.float32)
        pools.append(f32_to_bf16_bits(x) if dtype == "bf16" else x)
    return dict(slots=slots, num_accepted=acc, pools=pools, keep=keep, K=K, dtype=dtype)


def slot_copy_case(seed, P, n_src, fan_out, n_clear):
    """Disjoint parents, children and clears drawn from a P-slot pool."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(P).astype(np.int32)
    src = perm[:n_src]
    dst = perm[n_src:n_src + n_src * fan_out]
    clear = perm[n_src + n_src * fan_out:n_src + n_src * fan_out + n_clear]
    offs = (np.arange(n_src + 1) * fan_out).astype(np.int32)
    return dict(src=src, dst=dst, dst_offsets=offs, clear=clear)


# --------------------------------------------------------------------------
# the five serving workloads (sizes of the published configurations)

def tiny_prefill_512_h4():
    """1 sequence, T = 512, H = 4, fp32 throughout, S0 = 0, snapshot j = 3."""
    return prefill_case(0, [512], 4, dtype="f32", track=[[3]])


def batched_prefill_lengths(seed=1):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in rng.integers(1024, 8192 + 1, size=8)]


def batched_prefill_8seq_h32():
    """8 sequences, lengths ~ U[1024, 8192], H = 32, bf16, a 64-slot pool."""
    # lengths drawn first from the same stream, then slots, tracks, tokens, pool
    rng = np.random.Generator(np.random.PCG64(1))
    lengths = [int(x) for x in rng.integers(1024, 8192 + 1, size=8)]
    return _prefill_from_rng(rng, lengths, 32, "bf16", pool_slots=64)


def _prefill_from_rng(rng, lengths, H, dtype, pool_slots, dk=128, dv=128, chunk=64):
    N = len(lengths)
    cu = np.zeros(N + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    slots = rng.permutation(pool_slots)[:N].astype(np.int32)
    track = np.array([[rng.integers(0, (L + chunk - 1) // chunk)] for L in lengths], np.int32)
    tok = draw_tokens(rng, int(cu[-1]), H, dk, dv, dtype)
    pool = draw_pool(rng, pool_slots, H, dv, dk)
    return dict(tok, dtype=dtype, cu_seqlens=cu, N=N, T=int(cu[-1]), H=H, dk=dk, dv=dv,
                chunk=chunk, pool=pool, init_slot=slots, final_slot=slots, track=track,
                lengths=lengths)


def decode_256req_h32():
    """256 requests x 1 token, H = 32, bf16, a 1024-slot pool."""
    return decode_case(2, 256, 32, 1024)


def spec_64req_k7_h32():
    """Speculative verify + commit: 64 requests, K = 7, H = 32, bf16."""
    return spec_case(3, 64, 7, 32)


def long_prefill_131072_h16():
    """1 sequence, T = 131072, H = 16, snapshots every 64 chunks."""
    T = 131072
    track = [[64 * m for m in range(1, 32)]]
    return prefill_case(4, [T], 16, track=track, pool_slots=0)


def tp_slice_prefill_4x32768_h4():
    """4 sequences of 32768 tokens at H = 4 (a tensor-parallel slice of 32 heads), initial and
    final states in slots, one snapshot per sequence."""
    return prefill_case(14, [32768] * 4, 4, pool_slots=4, track_per_seq=1)


def slot_fanout_256x8_pool4096():
    """256 parents fanned out to 8 children each, plus 512 clears, in a 4096-slot pool."""
    return slot_copy_case(4, 4096, 256, 8, 512)
