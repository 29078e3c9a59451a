"""In-kernel q / k L2 normalisation (KDA_QK_L2NORM): every entry point that
reads q or k normalises each (row, head) in fp32 before use, and the commit
normalises the key record (which holds k as given).  Inputs here have rows of
arbitrary length, so the flag has to act; results are checked against the
fp64 oracle run with the same flag."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import TOL_STATE, dev_tensor, i32, rel_l2, to_np, worst_seq_head, worst_state

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


def _rescale_rows(c, seed):
    """q and k rows scaled by factors in [0.3, 4] (then rounded to bf16 again)."""
    rng = np.random.default_rng(seed)
    for name in ("q", "k"):
        x = W.bf16_bits_to_f32(c[name]).reshape(c[name].shape)
        f = rng.uniform(0.3, 4.0, x.shape[:-1] + (1,)).astype(np.float32)
        c[name] = W.f32_to_bf16_bits((x * f).astype(np.float32)).reshape(c[name].shape)
    return c


def _wid(c, n):
    return W.widen(c[n], "bf16")


@pytest.mark.parametrize("path", ["two_phase", "single_pass", "token_serial"])
def test_prefill(kda, path):
    c = _rescale_rows(W.prefill_case(80, [300, 1, 64, 777], 3, pool_slots=8, track_per_seq=2), 1)
    g = W.bf16_bits_to_f32(c["gate"]).copy()
    g[40:43, 1] = 40.0  # a chunk of head 1 that runs token by token
    c["gate"] = W.f32_to_bf16_bits(g)
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    pool = torch.from_numpy(c["pool"]).cuda()
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    snap = torch.full((N, M, H, 128, 128), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    if path == "two_phase":
        ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, N, H), dtype=torch.uint8, device="cuda")
    flags = kda.KDA_QK_L2NORM | (kda.KDA_PREFILL_RECURRENT if path == "token_serial" else 0)
    kda.kda_chunk_prefill(*(dev_tensor(c[n], "bf16") for n in ("q", "k", "v", "beta", "gate")),
                          i32(c["cu_seqlens"]), out, state_pool=pool, init_slot=i32(c["init_slot"]),
                          final_slot=i32(c["final_slot"]), track_chunk_idx=i32(c["track"]),
                          track_state=snap, dev_status=st, workspace=ws, flags=flags, scale=0.7)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S0 = c["pool"][c["init_slot"]].astype(np.float64)
    o_ref, s_ref, snap_ref, _ = oracle.prefill(_wid(c, "q"), _wid(c, "k"), _wid(c, "v"), _wid(c, "beta"),
                                               _wid(c, "gate"), c["cu_seqlens"], S0=S0, track=c["track"],
                                               flags=oracle.QK_L2NORM, scale=0.7)
    valid = c["track"] >= 0
    fin = pool.cpu().numpy()[c["final_slot"]]
    assert worst_seq_head(to_np(out), o_ref, c["cu_seqlens"]) < 5e-3
    assert worst_state(fin, s_ref) < TOL_STATE
    assert worst_state(snap.cpu().numpy()[valid], snap_ref[valid]) < TOL_STATE
    # without the flag the same inputs give a different answer: the rows are not unit length
    o_raw, _, _, _ = oracle.prefill(_wid(c, "q"), _wid(c, "k"), _wid(c, "v"), _wid(c, "beta"),
                                    _wid(c, "gate"), c["cu_seqlens"], S0=S0, scale=0.7)
    assert rel_l2(to_np(out), o_raw) > 0.05


def test_decode(kda):
    d = _rescale_rows(W.decode_case(81, 16, 4, 32), 2)
    pool = torch.from_numpy(d["pool"]).cuda()
    out = torch.empty(16, 4, 128, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_recurrent_decode(*(dev_tensor(d[n], "bf16") for n in ("q", "k", "v", "beta", "gate")),
                             pool, i32(d["slot"]), out, dev_status=st, flags=kda.KDA_QK_L2NORM)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, p_ref, _ = oracle.decode(_wid(d, "q"), _wid(d, "k"), _wid(d, "v"), _wid(d, "beta"),
                                    _wid(d, "gate"), d["pool"], d["slot"], flags=oracle.QK_L2NORM)
    assert rel_l2(to_np(out), o_ref) < 5e-3
    assert rel_l2(pool.cpu().numpy(), p_ref) < TOL_STATE


@pytest.mark.parametrize("K", [3, 7, 12])
def test_verify_then_commit(kda, K):
    R, H = 6, 4
    s = _rescale_rows(W.spec_case(82 + K, R, K, H), 3 + K)
    f = kda.KDA_QK_L2NORM
    pool = torch.from_numpy(s["pool"]).cuda()
    pool_fused = pool.clone()
    rec_u = torch.empty(R, H, K, 128, device="cuda")
    rec_kg = torch.empty(R, H, K, 256, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(R * K, H, 128, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc = W.accept_case(90 + K, R, K, p_match=0.7)
    a_ref, _, _ = oracle.accept(acc["tokens"], acc["sampled"], K)
    kda.kda_spec_verify(*(dev_tensor(s[n], "bf16") for n in ("q", "k", "v", "beta", "gate")),
                        pool, i32(s["ckpt"]), rec_u, rec_kg, out, K=K, dev_status=st, flags=f)
    kda.kda_spec_commit(pool, i32(s["ckpt"]), i32(a_ref), rec_u, rec_kg, K=K, dev_status=st, flags=f)
    kda.kda_spec_accept_commit(pool_fused, i32(s["ckpt"]), i32(acc["tokens"]), i32(acc["sampled"]),
                               rec_u, rec_kg, dev_status=st, flags=f)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, ru_ref, rkg_ref, _ = oracle.verify(_wid(s, "q"), _wid(s, "k"), _wid(s, "v"), _wid(s, "beta"),
                                              _wid(s, "gate"), s["pool"], s["ckpt"], K,
                                              flags=oracle.QK_L2NORM)
    assert rel_l2(to_np(out), o_ref) < 5e-3
    assert rel_l2(rec_u.cpu().numpy(), ru_ref) < TOL_STATE
    assert np.array_equal(to_np(rec_kg), rkg_ref)  # the key record holds k as given
    p_ref, _, _ = oracle.commit(s["pool"], s["ckpt"], a_ref, ru_ref, rkg_ref, K, flags=oracle.QK_L2NORM)
    assert worst_state(pool.cpu().numpy(), p_ref) < TOL_STATE
    assert torch.equal(pool_fused, pool)
