"""GPU parity of kda_spec_accept (integer work, bit-exact against the oracle)
and of the accept -> commit chain, which runs on one stream with no host
round trip between the two launches."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import TOL_STATE, dev_tensor, i32, rel_l2, tol_out, to_np, wid

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import serving_kda_chunk_gb300 as kda

    return kda


def _run_accept(kda, tokens, sampled, q_len, *, with_next=True):
    R = tokens.shape[0]
    acc = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")[:R]
    nxt = torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda")[:R] if with_next else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_spec_accept(i32(tokens), i32(sampled), acc,
                        q_len=None if q_len is None else i32(q_len),
                        next_token=nxt, dev_status=st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), None if nxt is None else nxt.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("K", [1, 2, 7, 16, 31, 32])
@pytest.mark.parametrize("p_match", [0.0, 0.7, 1.0])
def test_accept_bit_exact(kda, K, p_match):
    """301 requests (75 full four-warp CTAs and a ragged one), q_len drawn over
    [0, K] with a draftless and a padding row forced in."""
    R = 301
    rng = np.random.default_rng(1000 + K)
    ql = rng.integers(0, K + 1, size=R).astype(np.int32)
    ql[0], ql[1], ql[-1] = 1, 0, K
    c = W.accept_case(40 + K, R, K, q_len=ql, p_match=p_match)
    a, nxt, st = _run_accept(kda, c["tokens"], c["sampled"], c["q_len"])
    a_ref, n_ref, st_ref = oracle.accept(c["tokens"], c["sampled"], K, q_len=c["q_len"])
    assert st == st_ref == 0
    assert np.array_equal(a, a_ref)
    assert np.array_equal(nxt, n_ref)
    if p_match == 1.0:
        assert np.array_equal(a, ql)


def test_accept_defaults_and_bad_lengths(kda):
    K, R = 7, 9
    c = W.accept_case(50, R, K, p_match=0.8)
    # q_len omitted (= K), next_token omitted
    a, nxt, st = _run_accept(kda, c["tokens"], c["sampled"], None, with_next=False)
    a_ref, _, _ = oracle.accept(c["tokens"], c["sampled"], K)
    assert st == 0 and nxt is None and np.array_equal(a, a_ref)
    # out-of-range q_len: a = -1, next = -1 and the status bit; neighbours unaffected
    ql = np.array([7, -1, 8, 0, 1, 7, 1 << 30, -(1 << 30), 3], np.int32)
    a, nxt, st = _run_accept(kda, c["tokens"], c["sampled"], ql)
    a_ref, n_ref, st_ref = oracle.accept(c["tokens"], c["sampled"], K, q_len=ql)
    assert st == st_ref == kda.KDA_DEV_BAD_ACCEPT
    assert np.array_equal(a, a_ref) and np.array_equal(nxt, n_ref)
    assert a[1] == a[2] == a[6] == a[7] == -1
    # empty batch launches nothing
    empty = np.zeros((0, K), np.int32)
    a, nxt, st = _run_accept(kda, empty, empty, None)
    assert a.shape == (0,) and st == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_accept_commit_chain(kda, dtype):
    """verify -> accept -> commit on one stream, variable q_len with draftless
    (1) and padding (0) requests; the pool must equal the oracle's commit at
    the oracle's accepted lengths."""
    R, K, H, P = 24, 7, 2, 31
    rng = np.random.default_rng(77)
    ql = rng.integers(1, K + 1, size=R).astype(np.int32)
    ql[:3] = [1, 0, K]
    s = W.spec_case(60, R, K, H, P=P, dtype=dtype, q_len=ql)
    c = W.accept_case(61, R, K, q_len=ql, p_match=0.75)
    dt = s["dtype"]
    pool = torch.from_numpy(s["pool"]).cuda()
    rdt = torch.bfloat16 if dt == "bf16" else torch.float32
    rec_u = torch.empty(R, H, K, 128, device="cuda")
    rec_kg = torch.empty(R, H, K, 256, dtype=rdt, device="cuda")
    out = torch.empty(R * K, H, 128, dtype=rdt, device="cuda")
    acc = torch.empty(R, dtype=torch.int32, device="cuda")
    nxt = torch.empty(R, dtype=torch.int32, device="cuda")
    plan = torch.empty(R, 3, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ckpt, qlen = i32(s["ckpt"]), i32(ql)
    tokens, sampled = i32(c["tokens"]), i32(c["sampled"])
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        kda.kda_spec_verify(dev_tensor(s["q"], dt), dev_tensor(s["k"], dt), dev_tensor(s["v"], dt),
                            dev_tensor(s["beta"], dt), dev_tensor(s["gate"], dt), pool, ckpt,
                            rec_u, rec_kg, out, K=K, q_len=qlen, dev_status=st, stream=stream)
        kda.kda_spec_accept(tokens, sampled, acc, q_len=qlen, next_token=nxt, dev_status=st,
                            stream=stream)
        kda.kda_spec_commit(pool, ckpt, acc, rec_u, rec_kg, K=K, q_len=qlen, plan_out=plan,
                            dev_status=st, stream=stream)
    stream.synchronize()
    assert int(st.item()) == 0
    a_ref, n_ref, _ = oracle.accept(c["tokens"], c["sampled"], K, q_len=ql)
    assert np.array_equal(acc.cpu().numpy(), a_ref)
    assert np.array_equal(nxt.cpu().numpy(), n_ref)
    assert a_ref[0] == 1 and a_ref[1] == 0
    o_ref, ru_ref, rkg_ref, _ = oracle.verify(wid(s, "q"), wid(s, "k"), wid(s, "v"),
                                              wid(s, "beta"), wid(s, "gate"), s["pool"],
                                              s["ckpt"], K, q_len=ql)
    assert rel_l2(to_np(out), o_ref) < tol_out(dtype)
    p_ref, plan_ref, _ = oracle.commit(s["pool"], s["ckpt"], a_ref, ru_ref, rkg_ref, K, q_len=ql)
    assert np.array_equal(plan.cpu().numpy(), plan_ref)
    assert rel_l2(pool.cpu().numpy(), p_ref) < TOL_STATE
    # the padding request (a = 0, in place) leaves its checkpoint bit-identical
    assert np.array_equal(pool.cpu().numpy()[s["ckpt"][1]], s["pool"][s["ckpt"][1]])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_fused_accept_commit_matches_two_launches(kda, dtype):
    """kda_spec_accept_commit leaves the pool, plan, lengths, next tokens and
    status bit-identical to kda_spec_accept followed by kda_spec_commit, bad
    q_len and bad slots included, and matches the oracle."""
    R, K, H, P = 37, 5, 2, 50
    rng = np.random.default_rng(91)
    ql = rng.integers(0, K + 1, size=R).astype(np.int32)
    s = W.spec_case(90, R, K, H, P=P, dtype=dtype, q_len=np.clip(ql, 0, K))
    c = W.accept_case(92, R, K, q_len=np.clip(ql, 0, K), p_match=0.8)
    ql[4], ql[9] = K + 2, -3          # bad lengths: skipped, BAD_ACCEPT
    ckpt = s["ckpt"].copy()
    ckpt[13] = P + 1                  # bad slot: skipped, BAD_SLOT
    dst = ckpt.copy()
    dst[20] = sorted(set(range(P)) - set(s["ckpt"].tolist()))[0]  # one out-of-place commit
    dt = s["dtype"]
    rdt = torch.bfloat16 if dt == "bf16" else torch.float32
    pool0 = torch.from_numpy(s["pool"]).cuda()
    rec_u = torch.empty(R, H, K, 128, device="cuda")
    rec_kg = torch.empty(R, H, K, 256, dtype=rdt, device="cuda")
    out = torch.empty(R * K, H, 128, dtype=rdt, device="cuda")
    vq = i32(np.clip(ql, 0, K))
    st_v = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_spec_verify(dev_tensor(s["q"], dt), dev_tensor(s["k"], dt), dev_tensor(s["v"], dt),
                        dev_tensor(s["beta"], dt), dev_tensor(s["gate"], dt), pool0,
                        i32(s["ckpt"]), rec_u, rec_kg, out, K=K, q_len=vq, dev_status=st_v)
    tokens, sampled, qlen, ck, ds = (i32(c["tokens"]), i32(c["sampled"]), i32(ql), i32(ckpt),
                                     i32(dst))
    res = []
    for fused in (False, True):
        pool = pool0.clone()
        acc = torch.full((R,), -9, dtype=torch.int32, device="cuda")
        nxt = torch.full((R,), -9, dtype=torch.int32, device="cuda")
        plan = torch.full((R, 3), -9, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            kda.kda_spec_accept_commit(pool, ck, tokens, sampled, rec_u, rec_kg, dst_slot=ds,
                                       q_len=qlen, num_accepted=acc, next_token=nxt,
                                       plan_out=plan, dev_status=st)
        else:
            kda.kda_spec_accept(tokens, sampled, acc, q_len=qlen, next_token=nxt, dev_status=st)
            kda.kda_spec_commit(pool, ck, acc, rec_u, rec_kg, K=K, dst_slot=ds, q_len=qlen,
                                plan_out=plan, dev_status=st)
        torch.cuda.synchronize()
        res.append([x.cpu().numpy() for x in (pool, acc, nxt, plan, st)])
    assert int(st_v.item()) == 0
    for x, y in zip(*res):
        assert np.array_equal(x, y)
    pool, acc, nxt, plan, st = res[1]
    assert st[0] == kda.KDA_DEV_BAD_ACCEPT | kda.KDA_DEV_BAD_SLOT
    a_ref, n_ref, _ = oracle.accept(c["tokens"], c["sampled"], K, q_len=ql)
    assert np.array_equal(acc, a_ref) and np.array_equal(nxt, n_ref)
    _, ru_ref, rkg_ref, _ = oracle.verify(wid(s, "q"), wid(s, "k"), wid(s, "v"), wid(s, "beta"),
                                          wid(s, "gate"), s["pool"], s["ckpt"], K,
                                          q_len=np.clip(ql, 0, K))
    p_ref, plan_ref, st_ref = oracle.commit(s["pool"], ckpt, a_ref, ru_ref, rkg_ref, K, dst=dst,
                                            q_len=ql)
    assert np.array_equal(plan, plan_ref)
    assert st_ref == st[0]
    assert rel_l2(pool, p_ref) < TOL_STATE


def test_align_mode_boundary_states(kda):
    """Align mode: a request whose accepted span seq_len0+1 .. seq_len0+a holds
    a multiple of the block size also gets the state at that boundary (the
    commit at a_b = boundary - seq_len0) in its block slot; the block index
    after the step comes out for every request."""
    R, K, H, B = 16, 7, 2, 8
    P = 3 * R
    rng = np.random.default_rng(95)
    s = W.spec_case(96, R, K, H, P=P)
    c = W.accept_case(97, R, K, p_match=0.8)
    seq0 = rng.integers(0, 40, size=R).astype(np.int32)
    seq0[0], seq0[1] = 7, 1          # 7 + a crosses 8 for every a >= 1; 1 + a ends on 8 at a = 7
    free = np.array(sorted(set(range(P)) - set(s["ckpt"].tolist())), np.int32)
    block_slot = free[:R].copy()
    block_slot[2] = -1               # boundary state not wanted
    block_slot[3] = P + 5            # past the pool
    a_ref, _, _ = oracle.accept(c["tokens"], c["sampled"], K)
    a_b, idx = oracle.align_plan(seq0, a_ref, B)
    assert (a_b > 0).sum() >= 4, "the seeded spans should cross several boundaries"
    dt = "bf16"
    pool = torch.from_numpy(s["pool"]).cuda()
    rec_u = torch.empty(R, H, K, 128, device="cuda")
    rec_kg = torch.empty(R, H, K, 256, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(R * K, H, 128, dtype=torch.bfloat16, device="cuda")
    acc = torch.empty(R, dtype=torch.int32, device="cuda")
    bidx = torch.full((R,), -9, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_spec_verify(dev_tensor(s["q"], dt), dev_tensor(s["k"], dt), dev_tensor(s["v"], dt),
                        dev_tensor(s["beta"], dt), dev_tensor(s["gate"], dt), pool,
                        i32(s["ckpt"]), rec_u, rec_kg, out, K=K, dev_status=st)
    kda.kda_spec_accept_commit(pool, i32(s["ckpt"]), i32(c["tokens"]), i32(c["sampled"]), rec_u,
                               rec_kg, num_accepted=acc, seq_len0=i32(seq0), block_size=B,
                               block_slot=i32(block_slot), block_idx_out=bidx, dev_status=st)
    torch.cuda.synchronize()
    crossing3 = a_b[3] > 0
    assert int(st.item()) == (kda.KDA_DEV_BAD_SLOT if crossing3 else 0)
    assert np.array_equal(acc.cpu().numpy(), a_ref)
    assert np.array_equal(bidx.cpu().numpy(), idx)
    got = pool.cpu().numpy()
    _, ru_ref, rkg_ref, _ = oracle.verify(wid(s, "q"), wid(s, "k"), wid(s, "v"), wid(s, "beta"),
                                          wid(s, "gate"), s["pool"], s["ckpt"], K)
    run_ref, _, _ = oracle.commit(s["pool"], s["ckpt"], a_ref, ru_ref, rkg_ref, K)
    assert rel_l2(got[s["ckpt"]], run_ref[s["ckpt"]]) < TOL_STATE
    want_b = (a_b > 0) & (block_slot >= 0) & (block_slot < P)
    bnd_ref, _, _ = oracle.commit(s["pool"], s["ckpt"], np.where(want_b, a_b, 0), ru_ref, rkg_ref,
                                  K, dst=np.where(want_b, block_slot, s["ckpt"]))
    for r in range(R):
        if want_b[r]:
            assert rel_l2(got[block_slot[r]], bnd_ref[block_slot[r]]) < TOL_STATE, r
            if a_b[r] == a_ref[r]:  # the boundary is the end of the span: the same state
                assert np.array_equal(got[block_slot[r]], got[s["ckpt"][r]])
        elif 0 <= block_slot[r] < P:
            assert np.array_equal(got[block_slot[r]], s["pool"][block_slot[r]]), r
