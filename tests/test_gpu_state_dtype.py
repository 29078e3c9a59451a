"""GPU parity with bf16 / fp16 state pools (KDA_STATE_BF16 / KDA_STATE_F16).

Each entry point is checked three ways on the same seeded inputs:
  * against the fp64 oracle run on the widened 16-bit states, within the
    bound u + 1e-4 (u = unit roundoff of the state type: rounding moves every
    element by at most u relative, so the rel-L2 of the rounding error is at
    most u, on top of the fp32 tolerance);
  * exactly one rounding: the 16-bit result equals, bit for bit, the fp32
    path's result on the same widened inputs rounded once to nearest even;
  * outputs and records that do not pass through a state store are
    bit-identical to the fp32 path's.
A double-rounding probe writes, through decode, an fp32 value whose direct
fp16 rounding differs from its rounding through bf16."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import TOL_STATE, dev_tensor, i32, rel_l2, tol_out, to_np, wid

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

STATE_DTYPES = ["bf16", "f16"]
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import serving_kda_chunk_gb300 as kda

    return kda


def _tdt(sdt):
    return torch.bfloat16 if sdt == "bf16" else torch.float16


def _tol(sdt):
    return UNIT_ROUNDOFF[sdt] + TOL_STATE


def _narrow_pool(pool_f32, sdt):
    """(16-bit pool on the GPU, the same values widened to fp32 on the GPU,
    and widened to fp64 on the host for the oracle)."""
    p16 = torch.from_numpy(np.ascontiguousarray(pool_f32)).cuda().to(_tdt(sdt))
    p32 = p16.float()
    return p16, p32, p32.cpu().numpy().astype(np.float64)


def _same_bits(a16, b16):
    return torch.equal(a16.view(torch.int16), b16.view(torch.int16))


# --------------------------------------------------------------------------
# decode


@pytest.mark.parametrize("sdt", STATE_DTYPES)
def test_decode_16bit_pool(kda, sdt):
    d = W.decode_case(200, 37, 3, 50)
    p16, p32, p64 = _narrow_pool(d["pool"], sdt)
    args = [dev_tensor(d[n], "bf16") for n in ("q", "k", "v", "beta", "gate")]
    slot = i32(d["slot"])
    out16 = torch.empty(37, 3, 128, dtype=torch.bfloat16, device="cuda")
    out32 = torch.empty_like(out16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_recurrent_decode(*args, p16, slot, out16, dev_status=st)
    kda.kda_recurrent_decode(*args, p32, slot, out32, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out16, out32)
    assert _same_bits(p16, p32.to(_tdt(sdt)))
    o_ref, p_ref, _ = oracle.decode(wid(d, "q"), wid(d, "k"), wid(d, "v"), wid(d, "beta"),
                                    wid(d, "gate"), p64, d["slot"])
    assert rel_l2(to_np(out16), o_ref) < tol_out("bf16")
    assert rel_l2(p16.float().cpu().numpy(), p_ref) < _tol(sdt)


def test_fp16_pool_is_not_rounded_through_bf16(kda):
    """Zero state, alpha = 1, beta = 1, k = e_0: the new state's key-0 row is v
    exactly, so slot rows receive round(v).  v = 1 + 2^-8 + 2^-12 rounds to
    1 + 2^-8 in fp16 directly but to 1 + 2^-7 through bf16 first."""
    H, R = 1, 1
    x = np.float32(1.0 + 2.0 ** -8 + 2.0 ** -12)
    assert np.float16(x) == np.float16(1.0 + 2.0 ** -8)
    q = torch.zeros(R, H, 128, device="cuda")
    k = torch.zeros(R, H, 128, device="cuda")
    k[..., 0] = 1.0
    v = torch.full((R, H, 128), float(x), device="cuda")
    v[..., 1] = -float(x)
    beta = torch.ones(R, H, device="cuda")
    gate = torch.zeros(R, H, 128, device="cuda")
    flags = kda.KDA_GATE_LOG | kda.KDA_BETA_ACT
    for dt, want in ((torch.float16, 1.0 + 2.0 ** -8), (torch.bfloat16, 1.0 + 2.0 ** -7)):
        pool = torch.zeros(2, H, 128, 128, dtype=dt, device="cuda")
        out = torch.empty(R, H, 128, device="cuda")
        kda.kda_recurrent_decode(q, k, v, beta, gate, pool, i32([1]), out, flags=flags)
        torch.cuda.synchronize()
        row = pool[1, 0, :, 0].float().cpu().numpy()  # pool[slot][h][v][k]: key 0 of every v
        assert row[0] == want and row[1] == -want and (row[2:] == want).all()
        assert (pool[1, 0, :, 1:] == 0).all() and (pool[0] == 0).all()


# --------------------------------------------------------------------------
# prefill


def _run_prefill(kda, c, pool, snap_dtype, flags=0):
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    dt = c["dtype"]
    out = torch.full((max(T, 1), H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")[:T]
    snap = torch.zeros((N, M, H, 128, 128), dtype=snap_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_chunk_prefill(dev_tensor(c["q"], dt), dev_tensor(c["k"], dt), dev_tensor(c["v"], dt),
                          dev_tensor(c["beta"], dt), dev_tensor(c["gate"], dt),
                          i32(c["cu_seqlens"]), out, state_pool=pool,
                          init_slot=i32(c["init_slot"]), final_slot=i32(c["final_slot"]),
                          track_chunk_idx=i32(c["track"]), track_state=snap, flags=flags,
                          dev_status=st)
    torch.cuda.synchronize()
    return out, snap, int(st.item())


@pytest.mark.parametrize("sdt", STATE_DTYPES)
@pytest.mark.parametrize("path", ["tensor_core", "token_serial"])
def test_prefill_16bit_pool_and_snapshots(kda, sdt, path):
    lengths = [200, 64, 1, 130, 0]
    track = [[3, 1], [0, -1], [0, -1], [2, 0], [-1, -1]]
    c = W.prefill_case(210, lengths, 2, dtype="bf16", pool_slots=7, track=track)
    flags = kda.KDA_PREFILL_RECURRENT if path == "token_serial" else 0
    p16, p32, p64 = _narrow_pool(c["pool"], sdt)
    out16, snap16, st16 = _run_prefill(kda, c, p16, _tdt(sdt), flags)
    out32, snap32, st32 = _run_prefill(kda, c, p32, torch.float32, flags)
    assert st16 == st32 == 0
    assert torch.equal(out16, out32)
    assert _same_bits(p16, p32.to(_tdt(sdt)))
    assert _same_bits(snap16, snap32.to(_tdt(sdt)))
    S0 = np.stack([p64[s] for s in c["init_slot"]])
    o_ref, s_ref, snap_ref, _ = oracle.prefill(wid(c, "q"), wid(c, "k"), wid(c, "v"),
                                               wid(c, "beta"), wid(c, "gate"), c["cu_seqlens"],
                                               S0=S0, track=c["track"])
    assert rel_l2(to_np(out16), o_ref) < tol_out("bf16")
    fin = c["final_slot"]
    assert rel_l2(p16.float().cpu().numpy()[fin], s_ref) < _tol(sdt)
    valid = np.asarray(track) >= 0
    assert rel_l2(snap16.float().cpu().numpy()[valid], snap_ref[valid]) < _tol(sdt)
    # snapshot j = 0 is the initial state: widened and rounded back, it keeps the slot's bits
    init16 = torch.from_numpy(c["pool"][c["init_slot"][1]]).cuda().to(_tdt(sdt))
    assert _same_bits(snap16[1, 0], init16)


# --------------------------------------------------------------------------
# verify + commit


@pytest.mark.parametrize("sdt", STATE_DTYPES)
def test_verify_commit_16bit_pool(kda, sdt):
    R, K, H, P = 10, 7, 2, 14
    ql = np.array([7, 1, 0, 3, 7, 5, 2, 7, 6, 4], np.int32)
    s = W.spec_case(220, R, K, H, P=P, q_len=ql)
    c = W.accept_case(221, R, K, q_len=ql, p_match=0.7)
    p16, p32, p64 = _narrow_pool(s["pool"], sdt)
    args = [dev_tensor(s[n], "bf16") for n in ("q", "k", "v", "beta", "gate")]
    ckpt, qlen = i32(s["ckpt"]), i32(ql)
    dst = s["ckpt"].copy()
    dst[2] = sorted(set(range(P)) - set(s["ckpt"].tolist()))[0]  # a = 0 to another slot: a copy
    dsts = i32(dst)
    res = {}
    for name, pool in (("16", p16), ("32", p32)):
        rec_u = torch.empty(R, H, K, 128, device="cuda")
        rec_kg = torch.empty(R, H, K, 256, dtype=torch.bfloat16, device="cuda")
        out = torch.empty(R * K, H, 128, dtype=torch.bfloat16, device="cuda")
        acc = torch.empty(R, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda.kda_spec_verify(*args, pool, ckpt, rec_u, rec_kg, out, K=K, q_len=qlen, dev_status=st)
        kda.kda_spec_accept_commit(pool, ckpt, i32(c["tokens"]), i32(c["sampled"]), rec_u, rec_kg,
                                   dst_slot=dsts, q_len=qlen, num_accepted=acc, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        res[name] = (out, rec_u, rec_kg, acc)
    for a, b in zip(res["16"], res["32"]):
        assert torch.equal(a, b)  # verify reads the same widened values
    assert _same_bits(p16, p32.to(_tdt(sdt)))
    a_ref, _, _ = oracle.accept(c["tokens"], c["sampled"], K, q_len=ql)
    o_ref, ru_ref, rkg_ref, _ = oracle.verify(wid(s, "q"), wid(s, "k"), wid(s, "v"),
                                              wid(s, "beta"), wid(s, "gate"), p64, s["ckpt"], K,
                                              q_len=ql)
    out16, rec_u16, _, acc16 = res["16"]
    assert np.array_equal(acc16.cpu().numpy(), a_ref)
    assert rel_l2(to_np(out16), o_ref) < tol_out("bf16")
    assert rel_l2(rec_u16.cpu().numpy(), ru_ref) < TOL_STATE
    p_ref, _, _ = oracle.commit(p64, s["ckpt"], a_ref, ru_ref, rkg_ref, K, dst=dst, q_len=ql)
    assert rel_l2(p16.float().cpu().numpy(), p_ref) < _tol(sdt)
    # the padding request's checkpoint is copied to its destination bit for bit
    before = torch.from_numpy(s["pool"][s["ckpt"][2]]).cuda().to(_tdt(sdt))
    assert _same_bits(p16[dst[2]], before)
