"""The two-phase chunked prefill (a parallel prep over every (chunk, head), then a
sequential sweep per (sequence, head)), selected by a workspace of at least
kda_chunk_prefill_workspace_size bytes: parity with the fp64 oracle over ragged
lengths, the token path of chunks whose decay leaves the tensor-core range, fp32
outputs, fp32 activations (the chunk algorithm with fp32 inputs split into bf16
hi/lo operands), 16-bit state pools, the activation flags, snapshot placement,
and agreement with the single-pass and token-serial kernels."""
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


def run(kda, c, *, two_phase=True, flags=0, out_dtype=torch.bfloat16, ws_bytes=None):
    dt = c["dtype"]
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    pool = torch.from_numpy(c["pool"]).cuda()
    out = torch.full((T, H, 128), float("nan"), dtype=out_dtype, device="cuda")
    snap = torch.full((N, M, H, 128, 128), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    if two_phase:
        n = ws_bytes if ws_bytes is not None else kda.kda_chunk_prefill_workspace_size(T, N, H)
        ws = torch.empty(max(16, n), dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(dev_tensor(c["q"], dt), dev_tensor(c["k"], dt), dev_tensor(c["v"], dt),
                          dev_tensor(c["beta"], dt), dev_tensor(c["gate"], dt),
                          i32(c["cu_seqlens"]), out, state_pool=pool,
                          init_slot=i32(c["init_slot"]), final_slot=i32(c["final_slot"]),
                          track_chunk_idx=i32(c["track"]), track_state=snap, dev_status=st,
                          flags=flags, workspace=ws)
    torch.cuda.synchronize()
    return out, pool, snap, int(st.item())


def check(c, got, flags=0, tol_o=5e-3):
    out, pool, snap, st = got
    S0 = c["pool"][c["init_slot"]].astype(np.float64)
    dt = c["dtype"]
    o_ref, s_ref, snap_ref, _ = oracle.prefill(
        W.widen(c["q"], dt), W.widen(c["k"], dt), W.widen(c["v"], dt), W.widen(c["beta"], dt),
        W.widen(c["gate"], dt), c["cu_seqlens"], S0=S0, track=c["track"],
        flags=(flags & 3) | (oracle.QK_L2NORM if flags & 32 else 0))
    assert st == 0
    valid = c["track"] >= 0
    o = to_np(out)
    fin = pool.cpu().numpy()[c["final_slot"]]
    sn = snap.cpu().numpy()
    assert rel_l2(o, o_ref) < tol_o
    assert rel_l2(fin, s_ref) < TOL_STATE
    assert worst_seq_head(o, o_ref, c["cu_seqlens"]) < tol_o
    assert worst_state(fin, s_ref) < TOL_STATE
    if valid.any():
        assert rel_l2(sn[valid], snap_ref[valid]) < TOL_STATE
        assert worst_state(sn[valid], snap_ref[valid]) < TOL_STATE
    assert np.isnan(sn[~valid]).all()  # unused snapshot entries are never written
    return o, fin, sn


def test_ragged_lengths_and_snapshots(kda):
    lengths = [0, 1, 63, 64, 65, 200, 130, 1000]
    c = W.prefill_case(60, lengths, 3, pool_slots=16, track_per_seq=2)
    check(c, run(kda, c))


def test_one_long_sequence_few_heads(kda):
    c = W.prefill_case(61, [4096 + 17], 2, pool_slots=2, track_per_seq=4)
    check(c, run(kda, c))


def test_fp32_output(kda):
    c = W.prefill_case(62, [300, 77, 64], 2, pool_slots=6, track_per_seq=1)
    check(c, run(kda, c, out_dtype=torch.float32), tol_o=TOL_STATE)


@pytest.mark.parametrize("flags", [1, 2, 3])
def test_preactivated_flags(kda, flags):
    c = W.prefill_case(63, [150, 64], 2, pool_slots=4)
    if flags & 1:
        g = -np.abs(W.bf16_bits_to_f32(c["gate"])) * 0.5
        c["gate"] = W.f32_to_bf16_bits(g)
    if flags & 2:
        b = 1.0 / (1.0 + np.exp(-W.bf16_bits_to_f32(c["beta"])))
        c["beta"] = W.f32_to_bf16_bits(b.astype(np.float32))
    check(c, run(kda, c, flags=flags), flags=flags)


def test_strong_decay_chunks_take_the_token_path(kda):
    c = W.prefill_case(64, [256, 100], 2, pool_slots=4, track_per_seq=2)
    g = W.bf16_bits_to_f32(c["gate"]).copy()
    g[10:14] = 30.0        # chunk 0 of sequence 0, both heads
    g[200:203, 1] = 45.0   # chunk 3 of sequence 0, head 1 only
    g[300:302, 0] = 60.0   # the last (partial) chunk of sequence 1, head 0
    c["gate"] = W.f32_to_bf16_bits(g)
    check(c, run(kda, c))


def test_agrees_with_the_single_pass_kernel(kda):
    c = W.prefill_case(65, [700, 90, 1300], 4, pool_slots=6, track_per_seq=2)
    a = check(c, run(kda, c, two_phase=True))
    b = check(c, run(kda, c, two_phase=False))
    # the same arithmetic in a different order: far inside the oracle tolerances
    assert rel_l2(a[0], b[0]) < 5e-3 and rel_l2(a[1], b[1]) < 1e-5


def test_snapshot_placement_is_bit_exact(kda):
    # snapshot j of a full run == final state of a run over the first j*64 tokens
    L, j = 300, 3
    c = W.prefill_case(66, [L], 2, pool_slots=2, track=[[j, 0]])
    _, _, snap, st = run(kda, c)
    c2 = W.prefill_case(66, [L], 2, pool_slots=2, track=[[j, 0]])
    T2 = j * 64
    for key in ("q", "k", "v", "beta", "gate"):
        c2[key] = c2[key][:T2]
    c2["cu_seqlens"] = np.array([0, T2], np.int32)
    c2["T"] = T2
    c2["track"] = np.array([[0, -1]], np.int32)
    _, pool2, _, st2 = run(kda, c2)
    assert st == 0 and st2 == 0
    fin = int(c["final_slot"][0])
    assert torch.equal(snap[0, 0], pool2[fin])
    init = torch.from_numpy(c["pool"][c["init_slot"][0]]).cuda()
    assert torch.equal(snap[0, 1], init)


def test_deterministic(kda):
    c = W.prefill_case(67, [333, 64, 5], 2, pool_slots=6, track_per_seq=1)
    a = run(kda, c)
    b = run(kda, c)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x.nan_to_num(), y.nan_to_num())


def test_short_workspace_runs_the_single_pass_kernel(kda):
    c = W.prefill_case(68, [200, 50], 2, pool_slots=4)
    need = kda.kda_chunk_prefill_workspace_size(c["T"], c["N"], c["H"])
    a = run(kda, c, ws_bytes=need - 16)  # one byte short of the two-phase plan
    b = run(kda, c, two_phase=False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("st_flag", ["bf16", "f16"])
def test_16bit_state_pool(kda, st_flag):
    c = W.prefill_case(69, [260, 64], 2, pool_slots=4, track_per_seq=1)
    tdt = torch.bfloat16 if st_flag == "bf16" else torch.float16
    N, H, T = c["N"], c["H"], c["T"]
    pool = torch.from_numpy(c["pool"]).cuda().to(tdt)
    snap = torch.zeros((N, 1, H, 128, 128), dtype=tdt, device="cuda")
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, N, H), dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(*(dev_tensor(c[n], "bf16") for n in ("q", "k", "v", "beta", "gate")),
                          i32(c["cu_seqlens"]), out, state_pool=pool, init_slot=i32(c["init_slot"]),
                          final_slot=i32(c["final_slot"]), track_chunk_idx=i32(c["track"]),
                          track_state=snap, dev_status=st, workspace=ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S0 = pool.float().cpu().numpy()  # the widened 16-bit initial states
    wid = lambda n: W.widen(c[n], "bf16")  # noqa: E731
    o_ref, s_ref, snap_ref, _ = oracle.prefill(wid("q"), wid("k"), wid("v"), wid("beta"),
                                               wid("gate"), c["cu_seqlens"],
                                               S0=torch.from_numpy(c["pool"]).to(tdt).float()
                                               .numpy()[c["init_slot"]].astype(np.float64),
                                               track=c["track"])
    del S0
    u = 2.0 ** -8 if st_flag == "bf16" else 2.0 ** -11
    assert rel_l2(to_np(out), o_ref) < 5e-3
    assert rel_l2(pool.float().cpu().numpy()[c["final_slot"]], s_ref) < u + TOL_STATE
    valid = c["track"] >= 0
    assert rel_l2(snap.float().cpu().numpy()[valid], snap_ref[valid]) < u + TOL_STATE


# ---- fp32 activations: the same two kernels, the operands split from fp32 inputs


def test_fp32_activations_ragged_and_snapshots(kda):
    lengths = [0, 1, 63, 64, 65, 200, 130, 700]
    c = W.prefill_case(70, lengths, 3, dtype="f32", pool_slots=16, track_per_seq=2)
    check(c, run(kda, c, out_dtype=torch.float32), tol_o=TOL_STATE)


def test_fp32_activations_bf16_output(kda):
    c = W.prefill_case(71, [300, 77, 64], 2, dtype="f32", pool_slots=6, track_per_seq=1)
    check(c, run(kda, c, out_dtype=torch.bfloat16))


def test_fp32_activations_strong_decay_token_path(kda):
    c = W.prefill_case(72, [256, 100], 2, dtype="f32", pool_slots=4, track_per_seq=2)
    g = c["gate"].copy()
    g[10:14] = 30.0        # chunk 0 of sequence 0, both heads
    g[200:203, 1] = 45.0   # chunk 3 of sequence 0, head 1 only
    g[300:302, 0] = 60.0   # the last (partial) chunk of sequence 1, head 0
    c["gate"] = g
    check(c, run(kda, c, out_dtype=torch.float32), tol_o=TOL_STATE)


@pytest.mark.parametrize("flags", [1, 2])
def test_fp32_activations_preactivated_flags(kda, flags):
    c = W.prefill_case(73, [150, 64], 2, dtype="f32", pool_slots=4)
    if flags & 1:
        c["gate"] = (-np.abs(c["gate"]) * 0.5).astype(np.float32)
    if flags & 2:
        c["beta"] = (1.0 / (1.0 + np.exp(-c["beta"]))).astype(np.float32)
    check(c, run(kda, c, flags=flags, out_dtype=torch.float32), flags=flags, tol_o=TOL_STATE)


def test_fp32_activations_agree_with_token_serial(kda):
    # no workspace: fp32 activations run the token-serial kernel, the recurrence itself
    c = W.prefill_case(74, [500, 64, 3], 2, dtype="f32", pool_slots=6, track_per_seq=2)
    a = check(c, run(kda, c, two_phase=True, out_dtype=torch.float32), tol_o=TOL_STATE)
    b = check(c, run(kda, c, two_phase=False, out_dtype=torch.float32), tol_o=TOL_STATE)
    assert rel_l2(a[0], b[0]) < TOL_STATE and rel_l2(a[1], b[1]) < TOL_STATE


def test_fp32_activations_l2norm(kda):
    c = W.prefill_case(75, [300, 1, 64, 190], 3, dtype="f32", pool_slots=8, track_per_seq=2)
    rng = np.random.default_rng(75)
    for name in ("q", "k"):
        c[name] = (c[name] * rng.uniform(0.3, 4.0, c[name].shape[:-1] + (1,))).astype(np.float32)
    c["gate"][40:43, 1] = 40.0  # a chunk of head 1 that runs token by token
    flags = kda.KDA_QK_L2NORM
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    pool = torch.from_numpy(c["pool"]).cuda()
    out = torch.empty(T, H, 128, dtype=torch.float32, device="cuda")
    snap = torch.full((N, M, H, 128, 128), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, N, H), dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(*(dev_tensor(c[n], "f32") for n in ("q", "k", "v", "beta", "gate")),
                          i32(c["cu_seqlens"]), out, state_pool=pool, init_slot=i32(c["init_slot"]),
                          final_slot=i32(c["final_slot"]), track_chunk_idx=i32(c["track"]),
                          track_state=snap, dev_status=st, workspace=ws, flags=flags, scale=0.7)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S0 = c["pool"][c["init_slot"]].astype(np.float64)
    wid = lambda n: c[n].astype(np.float64)  # noqa: E731
    o_ref, s_ref, snap_ref, _ = oracle.prefill(wid("q"), wid("k"), wid("v"), wid("beta"), wid("gate"),
                                               c["cu_seqlens"], S0=S0, track=c["track"],
                                               flags=oracle.QK_L2NORM, scale=0.7)
    valid = c["track"] >= 0
    assert worst_seq_head(to_np(out), o_ref, c["cu_seqlens"]) < TOL_STATE
    assert worst_state(pool.cpu().numpy()[c["final_slot"]], s_ref) < TOL_STATE
    assert worst_state(snap.cpu().numpy()[valid], snap_ref[valid]) < TOL_STATE


# ---- edge cases of the plan: nothing to do, one head, the most snapshot requests


def test_all_sequences_empty(kda):
    # no tokens at all: the final states are the initial ones, bit for bit; nothing else written
    c = W.prefill_case(76, [0, 0, 0], 2, pool_slots=4, track_per_seq=1)
    assert c["T"] == 0 and (c["track"] == -1).all()
    out, pool, snap, st = run(kda, c)
    assert st == 0
    init = torch.from_numpy(c["pool"][c["init_slot"]]).cuda()
    assert torch.equal(pool[torch.from_numpy(c["final_slot"]).long().cuda()], init)
    assert torch.isnan(snap).all()


def test_single_head(kda):
    c = W.prefill_case(77, [300, 65, 1], 1, pool_slots=4, track_per_seq=2)
    check(c, run(kda, c))


@pytest.mark.parametrize("M", [512, 513])
def test_most_snapshot_requests(kda, M):
    # M = 512 is the two-phase plan's limit (duplicates and unused entries mixed); M = 513
    # takes the single-pass kernel with the same workspace
    track = np.full((1, M), -1, np.int32)
    track[0, [0, 100, 300, M - 1]] = [0, 2, 2, 4]
    c = W.prefill_case(78, [300], 1, pool_slots=2, track=track)
    check(c, run(kda, c))


def test_fp32_activations_bf16_state_pool(kda):
    c = W.prefill_case(79, [260, 64, 3], 2, dtype="f32", pool_slots=4, track_per_seq=1)
    N, H, T = c["N"], c["H"], c["T"]
    pool = torch.from_numpy(c["pool"]).cuda().to(torch.bfloat16)
    snap = torch.zeros((N, 1, H, 128, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(T, H, 128, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, N, H), dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(*(dev_tensor(c[n], "f32") for n in ("q", "k", "v", "beta", "gate")),
                          i32(c["cu_seqlens"]), out, state_pool=pool, init_slot=i32(c["init_slot"]),
                          final_slot=i32(c["final_slot"]), track_chunk_idx=i32(c["track"]),
                          track_state=snap, dev_status=st, workspace=ws, flags=kda.KDA_STATE_BF16)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S0 = torch.from_numpy(c["pool"]).to(torch.bfloat16).float().numpy()[c["init_slot"]].astype(np.float64)
    wid = lambda n: c[n].astype(np.float64)  # noqa: E731
    o_ref, s_ref, snap_ref, _ = oracle.prefill(wid("q"), wid("k"), wid("v"), wid("beta"), wid("gate"),
                                               c["cu_seqlens"], S0=S0, track=c["track"])
    u = 2.0 ** -8
    assert worst_seq_head(to_np(out), o_ref, c["cu_seqlens"]) < TOL_STATE
    assert worst_state(pool.float().cpu().numpy()[c["final_slot"]], s_ref) < u + TOL_STATE
    valid = c["track"] >= 0
    assert rel_l2(snap.float().cpu().numpy()[valid], snap_ref[valid]) < u + TOL_STATE


# ---- one long sequence with few heads.  With up to ~26 heads (on 152 SMs) the chunks are cut
#      into segments swept at once: every middle segment's state map Phi and offset B (the sweep
#      from S = I with V read as zero, and from S = 0), the segment start states chained from
#      them, then every segment swept from its start (2 heads x 256 chunks: 16 segments of 16).
#      With 27-38 heads the pipelined launches run instead (each segment's sweep beside the
#      prep of the next: [0, 8, 24, 56, 120, 248, 256) here).


def slow_decay(c, gate_shift=-8.0, beta_shift=-2.0):
    """Shift the raw gate and raw beta so that the state remembers across segments.  With the
    default recipe (raw gate ~ N(0,1): alpha ~ 1/2 per token) a segment's state map Phi is ~0
    and a wrong Phi or start state would go unseen; with alpha ~ 0.9997 and beta ~ 0.12 the
    start state still makes ~6 % of the state 16 chunks later (measured on the oracle)."""
    c = dict(c)
    for n, d in (("gate", gate_shift), ("beta", beta_shift)):
        x = W.widen(c[n], c["dtype"]).astype(np.float32) + np.float32(d)
        c[n] = W.store(x, c["dtype"])
    return c


def test_long_sequence_segment_scan_matches_oracle(kda):
    L = 256 * 64 - 17  # 256 chunks, the last one partial
    track = [[0, 15, 16, 17, 32, 100, 240, 255]]  # on, beside and between segment boundaries
    c = slow_decay(W.prefill_case(90, [L], 2, pool_slots=2, track=track))
    check(c, run(kda, c))


def test_long_sequence_segment_scan_fast_decay(kda):
    # the default recipe: Phi underflows towards zero, the start states come from B alone
    L = 256 * 64 - 17
    c = W.prefill_case(89, [L], 2, pool_slots=2, track=[[0, 16, 255]])
    check(c, run(kda, c))


def _as_first_of_two(c):
    """The same single sequence followed by an empty one: N = 2 takes the unsegmented launches."""
    L = c["lengths"][0]
    c2 = dict(c)
    c2["N"] = 2
    c2["cu_seqlens"] = np.array([0, L, L], np.int32)
    c2["init_slot"] = np.array([c["init_slot"][0], -1], np.int32)
    c2["final_slot"] = np.array([c["final_slot"][0], -1], np.int32)
    M = c["track"].shape[1]
    c2["track"] = np.concatenate([c["track"], np.full((1, M), -1, np.int32)])
    return c2


def test_long_sequence_segment_scan_close_to_unsegmented(kda):
    # the scan re-associates the state products (Phi_s S_s + B_s), so it agrees with the
    # unsegmented sweep to fp32 rounding rather than bit for bit
    L = 256 * 64 + 5
    c = slow_decay(W.prefill_case(93, [L], 3, pool_slots=2, track=[[3, 64, 250]]))
    a = run(kda, c)
    b = run(kda, _as_first_of_two(c))
    assert a[3] == 0 and b[3] == 0
    fin = int(c["final_slot"][0])
    assert rel_l2(to_np(a[0]), to_np(b[0])) < 1e-3  # bf16 outputs: a few last-bit flips
    assert rel_l2(a[1][fin].cpu().numpy(), b[1][fin].cpu().numpy()) < 1e-5
    assert rel_l2(a[2][0].cpu().numpy(), b[2][0].cpu().numpy()) < 1e-5


def test_long_sequence_segment_scan_deterministic(kda):
    c = slow_decay(W.prefill_case(94, [256 * 64], 2, pool_slots=2, track=[[5, 130]]))
    a = run(kda, c)
    b = run(kda, c)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_long_sequence_segment_scan_sequence_shorter_than_rows(kda):
    # 150 of 256 chunks' rows belong to the sequence: the segments past its end are skipped,
    # the segment holding its end writes the final state, and rows past it stay untouched
    L, R = 150 * 64 + 3, 256 * 64
    c = slow_decay(W.prefill_case(95, [L], 2, pool_slots=2, track=[[0, 16, 149]]))
    pad = W.prefill_case(96, [R - L], 2)
    cp = dict(c)
    for n in ("q", "k", "v", "beta", "gate"):
        cp[n] = np.concatenate([c[n], pad[n]])
    cp["T"] = R
    out, pool, snap, st = run(kda, cp)
    assert torch.isnan(out[L:].float()).all()
    check(c, (out[:L], pool, snap, st))


def test_long_sequence_segment_scan_strong_decay_token_path(kda):
    # chunks on the token path inside the Phi, B and output sweeps of middle segments
    L = 256 * 64
    c = slow_decay(W.prefill_case(97, [L], 2, pool_slots=2, track=[[40, 41, 200]]))
    g = W.bf16_bits_to_f32(c["gate"]).copy()
    g[40 * 64 + 10:40 * 64 + 14] = 30.0      # chunk 40, both heads (segment 2)
    g[41 * 64 + 3:41 * 64 + 5, 1] = 45.0     # chunk 41, head 1
    g[200 * 64 + 60:200 * 64 + 62, 0] = 60.0  # chunk 200, head 0 (segment 12)
    c["gate"] = W.f32_to_bf16_bits(g)
    check(c, run(kda, c))


def test_long_sequence_segment_scan_fp32_activations(kda):
    L = 256 * 64 + 30
    c = slow_decay(W.prefill_case(92, [L], 1, dtype="f32", pool_slots=2, track=[[0, 8, 100, 256]]))
    check(c, run(kda, c, out_dtype=torch.float32), tol_o=TOL_STATE)


@pytest.mark.parametrize("flags", [1, 2, 3])
def test_long_sequence_segment_scan_preactivated_flags(kda, flags):
    # the Phi and B sweeps with g given (KDA_GATE_LOG) and / or beta given (KDA_BETA_ACT), both
    # still slow to decay
    L = 256 * 64 - 5
    c = slow_decay(W.prefill_case(101, [L], 2, pool_slots=2, track=[[16, 130]]))
    if flags & 1:  # g = log alpha directly: alpha ~ 0.9995
        g = -np.abs(W.bf16_bits_to_f32(W.prefill_case(101, [L], 2)["gate"])) * np.float32(6e-4)
        c["gate"] = W.f32_to_bf16_bits(g.astype(np.float32))
    if flags & 2:  # beta itself, ~0.12
        b = 1.0 / (1.0 + np.exp(-W.bf16_bits_to_f32(c["beta"]).astype(np.float64)))
        c["beta"] = W.f32_to_bf16_bits(b.astype(np.float32))
    check(c, run(kda, c, flags=flags), flags=flags)


def test_long_sequence_segment_scan_l2norm(kda):
    # q and k rows of arbitrary length, normalised inside the kernels (KDA_QK_L2NORM)
    L = 256 * 64 + 7
    c = slow_decay(W.prefill_case(102, [L], 2, pool_slots=2, track=[[0, 100, 256]]))
    rng = np.random.default_rng(3)
    for n in ("q", "k"):
        x = W.bf16_bits_to_f32(c[n]).reshape(c[n].shape)
        f = rng.uniform(0.3, 4.0, x.shape[:-1] + (1,)).astype(np.float32)
        c[n] = W.f32_to_bf16_bits((x * f).astype(np.float32)).reshape(c[n].shape)
    check(c, run(kda, c, flags=kda.KDA_QK_L2NORM), flags=kda.KDA_QK_L2NORM)


def test_long_sequence_segment_scan_bf16_state_pool(kda):
    # start states, Phi and B stay fp32 in the workspace; only the final slot and the snapshots
    # round to bf16
    L = 256 * 64 - 70
    c = slow_decay(W.prefill_case(103, [L], 2, pool_slots=2, track=[[0, 17, 200]]))
    N, H, T = c["N"], c["H"], c["T"]
    pool = torch.from_numpy(c["pool"]).cuda().to(torch.bfloat16)
    snap = torch.zeros((N, 3, H, 128, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_chunk_prefill_workspace_size(T, N, H), dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(*(dev_tensor(c[n], "bf16") for n in ("q", "k", "v", "beta", "gate")),
                          i32(c["cu_seqlens"]), out, state_pool=pool, init_slot=i32(c["init_slot"]),
                          final_slot=i32(c["final_slot"]), track_chunk_idx=i32(c["track"]),
                          track_state=snap, dev_status=st, workspace=ws, flags=kda.KDA_STATE_BF16)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S0 = torch.from_numpy(c["pool"]).to(torch.bfloat16).float().numpy()[c["init_slot"]].astype(np.float64)
    wid = lambda n: W.widen(c[n], "bf16")  # noqa: E731
    o_ref, s_ref, snap_ref, _ = oracle.prefill(wid("q"), wid("k"), wid("v"), wid("beta"), wid("gate"),
                                               c["cu_seqlens"], S0=S0, track=c["track"])
    u = 2.0 ** -8
    assert worst_seq_head(to_np(out), o_ref, c["cu_seqlens"]) < 5e-3
    assert worst_state(pool.float().cpu().numpy()[c["final_slot"]], s_ref) < u + TOL_STATE
    assert worst_state(snap.float().cpu().numpy()[0], snap_ref[0]) < u + TOL_STATE


def test_long_sequence_segment_scan_fp32_output(kda):
    L = 256 * 64 - 40
    c = slow_decay(W.prefill_case(98, [L], 2, pool_slots=2, track=[[1, 47, 48]]))
    check(c, run(kda, c, out_dtype=torch.float32))


def test_several_long_sequences_segment_scan(kda):
    # two sequences of different lengths, 2 heads: the scan covers both, each unit's segments
    # cut from its own sequence's chunks
    lengths = [256 * 64 + 5, 300 * 64 - 7]
    c = slow_decay(W.prefill_case(104, lengths, 2, pool_slots=4, track=[[0, 100, 256], [17, 150, 299]]))
    check(c, run(kda, c))


def test_several_long_sequences_with_an_empty_and_a_short_one(kda):
    # four sequences, one empty and one of two chunks: segments of the short one are mostly
    # empty (identity maps, zero offsets), the empty one only carries its initial state to its
    # final slot
    lengths = [40000, 0, 30000, 70]
    track = [[0, 300], [-1, -1], [5, 400], [0, 1]]
    c = slow_decay(W.prefill_case(105, lengths, 2, pool_slots=6, track=track))
    check(c, run(kda, c))


def test_several_long_sequences_deterministic(kda):
    lengths = [256 * 64, 280 * 64 + 1]
    c = slow_decay(W.prefill_case(106, lengths, 2, pool_slots=4, track=[[9, 200], [3, 270]]))
    a = run(kda, c)
    b = run(kda, c)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_segment_scan_random_configurations(kda, seed):
    # seeded random draws inside the scan's range: 1-4 sequences of 16-40k tokens (one of them
    # possibly much shorter), 1-3 heads, random snapshot requests, the gate given as raw or as g
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 5))
    lengths = [int(x) for x in rng.integers(16384, 40000, N)]
    if N > 1 and rng.random() < 0.5:
        lengths[int(rng.integers(0, N))] = int(rng.integers(0, 3000))
    lengths[0] = max(lengths[0], 256 * 64 * N - sum(lengths[1:]))  # at least 256 chunks each on average
    H = int(rng.integers(1, 4))
    track = [[int(rng.integers(-1, (L + 63) // 64)) if L > 0 else -1 for _ in range(3)] for L in lengths]
    c = slow_decay(W.prefill_case(200 + seed, lengths, H, pool_slots=N + 1, track=track))
    flags = 0
    if rng.random() < 0.5:  # the gate as g = log alpha, slow decay
        g = -np.abs(W.bf16_bits_to_f32(W.prefill_case(200 + seed, lengths, H)["gate"])) * np.float32(6e-4)
        c["gate"] = W.f32_to_bf16_bits(g.astype(np.float32))
        flags = kda.KDA_GATE_LOG
    check(c, run(kda, c, flags=flags), flags=flags)


def test_long_sequence_pipelined_matches_oracle(kda):
    L = 256 * 64 - 17
    track = [[0, 8, 9, 24, 57, 200, 255]]  # on, beside and between segment boundaries
    c = slow_decay(W.prefill_case(99, [L], 32, pool_slots=2, track=track))
    check(c, run(kda, c))


def test_long_sequence_pipelined_bit_exact(kda):
    # the segments hand the fp32 state over exactly, so every result is bit-identical to the
    # unsegmented launches
    L = 256 * 64 + 5
    c = slow_decay(W.prefill_case(91, [L], 32, pool_slots=2, track=[[3, 64, 250]]))
    a = run(kda, c)
    b = run(kda, _as_first_of_two(c))
    assert a[3] == 0 and b[3] == 0
    assert torch.equal(a[0], b[0])
    fin = int(c["final_slot"][0])
    assert torch.equal(a[1][fin], b[1][fin])
    assert torch.equal(a[2][0], b[2][0])


def test_long_sequence_pipelined_fp32_activations(kda):
    # the combined launch with fp32 activations (its prep role at 96 registers)
    L = 256 * 64 + 30
    c = slow_decay(W.prefill_case(100, [L], 32, dtype="f32", pool_slots=2, track=[[0, 8, 100, 256]]))
    check(c, run(kda, c, out_dtype=torch.float32), tol_o=TOL_STATE)
