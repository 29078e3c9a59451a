"""GPU parity: every entry point through the C ABI against the fp64 oracle on
small seeded inputs that still span several tiles and ragged tails, plus the
edge cases of the method (empty and one-token sequences, snapshots at the
first and last chunk, accepted length 0 and K, padding slots, bad indices)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import (TOL_STATE, dev_tensor, i32, rel_l2, tol_out, to_np, wid, worst_seq_head,
                     worst_state)

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


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# --------------------------------------------------------------------------
# prefill


def run_prefill(kda, c, out_dtype=None, init=True, workspace=False):
    dt = c["dtype"]
    odt = out_dtype or (torch.bfloat16 if dt == "bf16" else torch.float32)
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    pool = torch.from_numpy(c["pool"]).cuda() if c["pool"] is not None else None
    out = torch.full((max(T, 1), H, 128), float("nan"), dtype=odt, device="cuda")[:T]
    snap = torch.full((N, M, H, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = _status()
    ws = None
    if workspace:  # the two-phase chunk path (bf16 or fp32 activations)
        ws = torch.empty(max(16, kda.kda_chunk_prefill_workspace_size(T, N, H)), dtype=torch.uint8,
                         device="cuda")
    kda.kda_chunk_prefill(dev_tensor(c["q"], dt), dev_tensor(c["k"], dt), dev_tensor(c["v"], dt),
                          dev_tensor(c["beta"], dt), dev_tensor(c["gate"], dt),
                          i32(c["cu_seqlens"]), out, state_pool=pool,
                          init_slot=i32(c["init_slot"]) if init else None,
                          final_slot=i32(c["final_slot"]), track_chunk_idx=i32(c["track"]),
                          track_state=snap, dev_status=st, workspace=ws)
    torch.cuda.synchronize()
    return out, pool, snap, int(st.item())


def oracle_prefill(c, init=True):
    S0 = None
    if c["pool"] is not None and init:
        S0 = np.stack([c["pool"][s] if s >= 0 else np.zeros(c["pool"].shape[1:], np.float32)
                       for s in c["init_slot"]]).astype(np.float64)
    return oracle.prefill(wid(c, "q"), wid(c, "k"), wid(c, "v"), wid(c, "beta"), wid(c, "gate"),
                          c["cu_seqlens"], S0=S0, track=c["track"])


@pytest.mark.parametrize("workspace", [False, True], ids=["no_workspace", "workspace"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefill_ragged_small(kda, dtype, workspace):
    # without a workspace: single-pass (bf16) or token-serial (f32); with one: two-phase chunks
    lengths = [0, 1, 63, 64, 65, 200, 130]
    track = [[-1, -1], [0, -1], [0, -1], [0, -1], [1, 0], [3, 1], [2, -1]]
    c = W.prefill_case(7, lengths, 3, dtype=dtype, pool_slots=12, track=track)
    out, pool, snap, st = run_prefill(kda, c, workspace=workspace)
    o_ref, s_ref, snap_ref, st_ref = oracle_prefill(c)
    assert st == 0 and st_ref == 0
    assert rel_l2(to_np(out), o_ref) < tol_out(dtype)
    assert rel_l2(pool.cpu().numpy()[c["final_slot"]], s_ref) < TOL_STATE
    valid = np.asarray(track) >= 0
    sn = snap.cpu().numpy()
    assert rel_l2(sn[valid], snap_ref[valid]) < TOL_STATE
    assert np.isnan(sn[~valid]).all()  # unused entries are never written
    # per (sequence, head), every ragged length on its own
    assert worst_seq_head(to_np(out), o_ref, c["cu_seqlens"]) < tol_out(dtype)
    assert worst_state(pool.cpu().numpy()[c["final_slot"]], s_ref) < TOL_STATE
    assert worst_state(sn[valid], snap_ref[valid]) < TOL_STATE


def test_prefill_zero_initial_state_and_fp32_output(kda):
    c = W.prefill_case(8, [100, 37], 2, dtype="bf16", pool_slots=4, with_init=False,
                       track_per_seq=2)
    out, pool, snap, st = run_prefill(kda, c, out_dtype=torch.float32, init=False)
    o_ref, s_ref, snap_ref, _ = oracle_prefill(c, init=False)
    assert st == 0
    # fp32 output of bf16 inputs: the result is not rounded, so hold it to the state tolerance
    assert rel_l2(to_np(out), o_ref) < TOL_STATE
    assert rel_l2(pool.cpu().numpy()[c["final_slot"]], s_ref) < TOL_STATE


def test_snapshot_placement_is_bit_exact(kda):
    # snapshot j of a full run == final state of a run over the first j*64 tokens (same kernel)
    L, j = 300, 3
    c = W.prefill_case(9, [L], 2, pool_slots=2, track=[[j, 0]])
    out, pool, snap, st = run_prefill(kda, c)
    c2 = W.prefill_case(9, [L], 2, pool_slots=2, track=[[j, 0]])
    T2 = j * 64
    for key in ("q", "k", "v", "beta", "gate"):
        c2[key] = c2[key][:T2]
    c2["cu_seqlens"] = np.array([0, T2], np.int32)
    c2["T"] = T2
    c2["track"] = np.array([[0, -1]], np.int32)
    _, pool2, snap2, _ = run_prefill(kda, c2)
    fin = int(c["final_slot"][0])
    assert torch.equal(snap[0, 0], pool2[fin])
    # j = 0 is the initial state, copied exactly
    init = torch.from_numpy(c["pool"][c["init_slot"][0]]).cuda()
    assert torch.equal(snap[0, 1], init) and torch.equal(snap2[0, 0], init)


def test_prefill_is_deterministic(kda):
    c = W.prefill_case(10, [150, 77], 2, pool_slots=4)
    a = run_prefill(kda, c)
    b = run_prefill(kda, c)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_prefill_reports_bad_indices(kda):
    # bad track index (>= n_chunks): reported, snapshot not written, rest computed
    c = W.prefill_case(11, [100], 1, pool_slots=2, track=[[2, 1]])
    out, pool, snap, st = run_prefill(kda, c)
    assert st & kda.KDA_DEV_BAD_TRACK
    assert torch.isnan(snap[0, 0]).all() and not torch.isnan(snap[0, 1]).any()
    # non-monotone cu_seqlens: the sequence is skipped and reported
    c = W.prefill_case(12, [10, 10], 1, pool_slots=2)
    c["cu_seqlens"] = np.array([0, 15, 12], np.int32)
    _, _, _, st = run_prefill(kda, c)
    assert st & kda.KDA_DEV_BAD_SEQLEN
    # final slot past the pool
    c = W.prefill_case(13, [10], 1, pool_slots=2)
    c["final_slot"] = np.array([5], np.int32)
    _, _, _, st = run_prefill(kda, c)
    assert st & kda.KDA_DEV_BAD_SLOT


def test_prefill_special_gates_identity(kda):
    # raw gate -inf (alpha = 1) and raw beta -inf (beta = 0): the state is unchanged exactly
    c = W.prefill_case(14, [90], 2, dtype="f32", pool_slots=2)
    c["gate"] = np.full_like(c["gate"], -np.inf)
    c["beta"] = np.full_like(c["beta"], -np.inf)
    out, pool, _, st = run_prefill(kda, c)
    assert st == 0
    s0 = c["pool"][c["init_slot"][0]]
    assert np.array_equal(pool.cpu().numpy()[c["final_slot"][0]], s0)


# --------------------------------------------------------------------------
# decode


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_small(kda, dtype):
    d = W.decode_case(20, 9, 3, 20, dtype=dtype, skip=(4,))
    pool = torch.from_numpy(d["pool"]).cuda()
    odt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.full((9, 3, 128), float("nan"), dtype=odt, device="cuda")
    st = _status()
    kda.kda_recurrent_decode(dev_tensor(d["q"], dtype), dev_tensor(d["k"], dtype),
                             dev_tensor(d["v"], dtype), dev_tensor(d["beta"], dtype),
                             dev_tensor(d["gate"], dtype), pool, i32(d["slot"]), out,
                             dev_status=st)
    torch.cuda.synchronize()
    o_ref, p_ref, _ = oracle.decode(wid(d, "q"), wid(d, "k"), wid(d, "v"), wid(d, "beta"),
                                    wid(d, "gate"), d["pool"], d["slot"])
    assert int(st.item()) == 0
    assert rel_l2(to_np(out), o_ref) < tol_out(dtype)
    assert (out[4] == 0).all()
    assert rel_l2(pool.cpu().numpy(), p_ref) < TOL_STATE
    untouched = sorted(set(range(20)) - set(d["slot"].tolist()))
    assert np.array_equal(pool.cpu().numpy()[untouched], d["pool"][untouched])


def test_decode_bad_slot(kda):
    d = W.decode_case(21, 2, 1, 4)
    d["slot"] = np.array([7, 1], np.int32)
    pool = torch.from_numpy(d["pool"]).cuda()
    out = torch.full((2, 1, 128), 1.0, dtype=torch.bfloat16, device="cuda")
    st = _status()
    kda.kda_recurrent_decode(dev_tensor(d["q"], "bf16"), dev_tensor(d["k"], "bf16"),
                             dev_tensor(d["v"], "bf16"), dev_tensor(d["beta"], "bf16"),
                             dev_tensor(d["gate"], "bf16"), pool, i32(d["slot"]), out,
                             dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kda.KDA_DEV_BAD_SLOT
    assert (out[0] == 0).all()


# --------------------------------------------------------------------------
# verify + commit


def run_verify(kda, s, out_dtype=None):
    dt = s["dtype"]
    R, K, H = s["R"], s["K"], s["H"]
    pool = torch.from_numpy(s["pool"]).cuda()
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    rec_u = torch.full((R, H, K, 128), float("nan"), device="cuda")
    rec_kg = torch.full((R, H, K, 256), float("nan"), dtype=tdt, device="cuda")
    out = torch.full((R * K, H, 128), float("nan"), dtype=out_dtype or tdt, device="cuda")
    st = _status()
    kda.kda_spec_verify(dev_tensor(s["q"], dt), dev_tensor(s["k"], dt), dev_tensor(s["v"], dt),
                        dev_tensor(s["beta"], dt), dev_tensor(s["gate"], dt), pool,
                        i32(s["ckpt"]), rec_u, rec_kg, out, K=K, q_len=i32(s["q_len"]),
                        dev_status=st)
    torch.cuda.synchronize()
    return pool, rec_u, rec_kg, out, int(st.item())


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_verify_then_commit_small(kda, dtype):
    R, K, H = 6, 4, 2
    s = W.spec_case(30, R, K, H, P=9, dtype=dtype, q_len=[4, 1, 0, 3, 4, 2])
    s["num_accepted"] = np.array([4, 0, 0, 2, 1, 2], np.int32)
    pool, rec_u, rec_kg, out, st = run_verify(kda, s)
    assert st == 0
    o_ref, ru_ref, rkg_ref, _ = oracle.verify(wid(s, "q"), wid(s, "k"), wid(s, "v"),
                                              wid(s, "beta"), wid(s, "gate"), s["pool"],
                                              s["ckpt"], K, q_len=s["q_len"])
    assert rel_l2(to_np(out), o_ref) < tol_out(dtype)
    assert rel_l2(rec_u.cpu().numpy(), ru_ref) < TOL_STATE
    # key / raw gate records are the input bits, zero past q_len
    assert np.array_equal(to_np(rec_kg), rkg_ref)
    assert np.array_equal(pool.cpu().numpy(), s["pool"])  # verify never writes the pool
    # commit in place, one request to another slot
    dst = s["ckpt"].copy()
    free = sorted(set(range(9)) - set(s["ckpt"].tolist()))
    dst[1] = free[0]
    plan = torch.zeros(R, 3, dtype=torch.int32, device="cuda")
    st_t = _status()
    kda.kda_spec_commit(pool, i32(s["ckpt"]), i32(s["num_accepted"]), rec_u, rec_kg, K=K,
                        dst_slot=i32(dst), q_len=i32(s["q_len"]), plan_out=plan, dev_status=st_t)
    torch.cuda.synchronize()
    assert int(st_t.item()) == 0
    want_plan = oracle.commit_plan(s["ckpt"], s["num_accepted"], 9, K, dst=dst, q_len=s["q_len"])
    assert np.array_equal(plan.cpu().numpy(), want_plan)
    # primary: brute-force recursion on the oracle's own records
    p_ref, _, _ = oracle.commit(s["pool"], s["ckpt"], s["num_accepted"], ru_ref, rkg_ref, K,
                                dst=dst, q_len=s["q_len"])
    assert rel_l2(pool.cpu().numpy(), p_ref) < TOL_STATE
    # same recursion on the GPU's recorded u: isolates the commit arithmetic
    p_ref2, _, _ = oracle.commit(s["pool"], s["ckpt"], s["num_accepted"],
                                 rec_u.cpu().numpy(), to_np(rec_kg), K, dst=dst,
                                 q_len=s["q_len"])
    assert rel_l2(pool.cpu().numpy(), p_ref2) < 1e-6
    # a = 0 to another slot is an exact copy
    assert np.array_equal(pool.cpu().numpy()[dst[1]], s["pool"][s["ckpt"][1]])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K", [2, 8, 16])
def test_verify_strong_decay_and_k_bounds(kda, K, dtype):
    # request 1 decays by ~e^-25 per step: its mid-reference factors leave the range the
    # verify pair tables carry (> 2^64 over K/2 steps for K >= 4), so that unit takes the
    # reduce-scatter path; the others take the table path in the same launch
    R, H = 4, 2
    s = W.spec_case(34 + K, R, K, H, P=6, dtype=dtype)
    gate = s["gate"].copy()
    strong = np.full(gate[K:2 * K].shape, 25.0, np.float32)
    gate[K:2 * K] = W.f32_to_bf16_bits(strong) if dtype == "bf16" else strong
    s["gate"] = gate
    pool, rec_u, rec_kg, out, st = run_verify(kda, s)
    assert st == 0
    o_ref, ru_ref, rkg_ref, _ = oracle.verify(wid(s, "q"), wid(s, "k"), wid(s, "v"),
                                              wid(s, "beta"), wid(s, "gate"), s["pool"],
                                              s["ckpt"], K, q_len=s["q_len"])
    assert rel_l2(to_np(out), o_ref) < tol_out(dtype)
    assert rel_l2(rec_u.cpu().numpy(), ru_ref) < TOL_STATE
    assert np.array_equal(to_np(rec_kg), rkg_ref)


def test_commit_rejects_bad_accept(kda):
    s = W.spec_case(31, 3, 3, 1, P=4)
    pool, rec_u, rec_kg, _, _ = run_verify(kda, s)
    acc = np.array([4, 1, -1], np.int32)
    plan = torch.zeros(3, 3, dtype=torch.int32, device="cuda")
    st = _status()
    before = pool.clone()
    kda.kda_spec_commit(pool, i32(s["ckpt"]), i32(acc), rec_u, rec_kg, K=3, plan_out=plan,
                        dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kda.KDA_DEV_BAD_ACCEPT
    pl = plan.cpu().numpy()
    assert pl[0, 0] == -1 and pl[2, 0] == -1 and pl[1, 0] == 1
    for r in (0, 2):
        c = int(s["ckpt"][r])
        assert torch.equal(pool[c], before[c])


def test_verify_accept_all_equals_decode_steps(kda):
    # verify + commit(a = K) == K decode steps on the same slot (both on the GPU, vs oracle)
    R, K, H = 2, 5, 2
    s = W.spec_case(32, R, K, H, P=2)
    pool, rec_u, rec_kg, out, _ = run_verify(kda, s)
    acc = np.full(R, K, np.int32)
    kda.kda_spec_commit(pool, i32(s["ckpt"]), i32(acc), rec_u, rec_kg, K=K)
    dpool = torch.from_numpy(s["pool"]).cuda()
    for t in range(K):
        rows = np.arange(R) * K + t
        sl = lambda n: dev_tensor(np.ascontiguousarray(s[n][rows]), "bf16")  # noqa: E731
        dout = torch.empty(R, H, 128, dtype=torch.bfloat16, device="cuda")
        kda.kda_recurrent_decode(sl("q"), sl("k"), sl("v"), sl("beta"), sl("gate"), dpool,
                                 i32(s["ckpt"]), dout)
        assert rel_l2(to_np(dout), to_np(out[rows])) < 5e-3
    torch.cuda.synchronize()
    assert rel_l2(pool.cpu().numpy(), dpool.cpu().numpy()) < TOL_STATE


# --------------------------------------------------------------------------
# slot copy


def run_copy(kda, pools, sc):
    maxs = max(p.shape[0] for p in pools)
    ws = torch.empty(kda.kda_slot_copy_workspace_size(maxs), dtype=torch.uint8, device="cuda")
    st = _status()
    kda.kda_slot_copy(pools, i32(sc["clear"]), i32(sc["src"]), i32(sc["dst_offsets"]),
                      i32(sc["dst"]), ws, dev_status=st)
    torch.cuda.synchronize()
    return int(st.item())


def test_slot_copy_multi_pool_fan_out(kda):
    sc = W.slot_copy_case(40, 50, 5, 3, 7)
    g = torch.Generator(device="cpu").manual_seed(0)
    pools = [torch.randn(50, 2, 128, 128, generator=g).cuda(),
             torch.randn(50, 3, 4, 4, generator=g).cuda(),        # 192 B slots: ragged piece
             torch.randint(0, 255, (50, 4000), dtype=torch.uint8, generator=g).cuda()[:, :3984]
             .contiguous()]
    before = [p.cpu().numpy() for p in pools]
    st = run_copy(kda, pools, sc)
    assert st == 0
    want = oracle.slot_copy(before, sc["clear"], sc["src"], sc["dst_offsets"], sc["dst"])
    for p, w in zip(pools, want):
        assert np.array_equal(p.cpu().numpy(), w)


def test_slot_copy_strided_pool(kda):
    # slots that are views into a larger per-slot record (stride > slot bytes)
    big = torch.randn(20, 2, 64, device="cuda")
    view = big[:, 0]
    sc = W.slot_copy_case(41, 20, 2, 2, 3)
    maxs = 20
    ws = torch.empty(kda.kda_slot_copy_workspace_size(maxs), dtype=torch.uint8, device="cuda")
    desc = (kda.PoolDesc * 1)()
    desc[0] = kda.PoolDesc(view.data_ptr(), big.stride(0) * 4, 64 * 4, 20)
    before = big.cpu().numpy()
    L = kda.lib()
    # keep the index tensors alive until the launch has completed
    clear, src, offs, dst = (i32(sc[n]) for n in ("clear", "src", "dst_offsets", "dst"))
    st = L.kda_slot_copy(desc, 1, clear.data_ptr(), 3, src.data_ptr(), offs.data_ptr(),
                         dst.data_ptr(), 2, 4, ws.data_ptr(), ws.numel(), None,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    (want,) = oracle.slot_copy([before[:, 0]], sc["clear"], sc["src"], sc["dst_offsets"],
                               sc["dst"])
    after = big.cpu().numpy()
    assert np.array_equal(after[:, 0], want)
    assert np.array_equal(after[:, 1], before[:, 1])  # bytes between slots untouched


@pytest.mark.parametrize("case", ["dup_dst", "src_is_dst", "clear_is_src", "out_of_range"])
def test_slot_copy_rejects_overlap(kda, case):
    sc = W.slot_copy_case(42, 30, 3, 2, 2)
    if case == "dup_dst":
        sc["dst"][1] = sc["dst"][0]
    elif case == "src_is_dst":
        sc["dst"][2] = sc["src"][0]
    elif case == "clear_is_src":
        sc["clear"][0] = sc["src"][1]
    else:
        sc["dst"][0] = 30
    pool = torch.randn(30, 64, device="cuda")
    before = pool.clone()
    st = run_copy(kda, [pool], sc)
    bit = kda.KDA_DEV_BAD_SLOT if case == "out_of_range" else kda.KDA_DEV_OVERLAP
    assert st & bit
    assert torch.equal(pool, before)  # nothing copied


def test_slot_copy_empty_sets(kda):
    pool = torch.randn(8, 64, device="cuda")
    before = pool.clone()
    sc = dict(clear=np.zeros(0, np.int32), src=np.zeros(0, np.int32),
              dst_offsets=np.zeros(1, np.int32), dst=np.zeros(0, np.int32))
    ws = torch.empty(kda.kda_slot_copy_workspace_size(8), dtype=torch.uint8, device="cuda")
    kda.kda_slot_copy([pool], None, None, i32(sc["dst_offsets"]), None, ws)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)
