"""The single-pass tensor-core chunked prefill (no workspace, or one too small
for the two-phase plan): parity with the fp64 oracle across chunk boundaries,
its large-decay fallback, the activation flags, the longest-first schedule, and
the chunk-vs-recurrent numerical gap (reported, and bounded)."""
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


def run(kda, c, flags=0, workspace=False, out_dtype=torch.bfloat16):
    dt = c["dtype"]
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    pool = torch.from_numpy(c["pool"]).cuda()
    out = torch.empty(T, H, 128, dtype=out_dtype, device="cuda")
    snap = torch.full((N, M, H, 128, 128), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    if workspace:
        # one byte short of the two-phase plan: the single-pass kernel with its
        # longest-first order (the two-phase path has its own tests)
        ws = torch.empty(max(16, kda.kda_chunk_prefill_workspace_size(T, N, H) - 16),
                         dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prefill(dev_tensor(c["q"], dt), dev_tensor(c["k"], dt), dev_tensor(c["v"], dt),
                          dev_tensor(c["beta"], dt), dev_tensor(c["gate"], dt),
                          i32(c["cu_seqlens"]), out, state_pool=pool,
                          init_slot=i32(c["init_slot"]), final_slot=i32(c["final_slot"]),
                          track_chunk_idx=i32(c["track"]), track_state=snap, dev_status=st,
                          flags=flags, workspace=ws)
    torch.cuda.synchronize()
    return out, pool, snap, int(st.item())


def ref(c, flags=0):
    dt = c["dtype"]
    S0 = c["pool"][c["init_slot"]].astype(np.float64)
    return oracle.prefill(W.widen(c["q"], dt), W.widen(c["k"], dt), W.widen(c["v"], dt),
                          W.widen(c["beta"], dt), W.widen(c["gate"], dt), c["cu_seqlens"], S0=S0,
                          track=c["track"], flags=flags)


def check(c, got, flags=0, tol_o=5e-3):
    out, pool, snap, st = got
    o_ref, s_ref, snap_ref, _ = ref(c, flags & 3)
    assert st == 0
    eo = rel_l2(to_np(out), o_ref)
    es = rel_l2(pool.cpu().numpy()[c["final_slot"]], s_ref)
    valid = c["track"] >= 0
    en = rel_l2(snap.cpu().numpy()[valid], snap_ref[valid]) if valid.any() else 0.0
    assert eo < tol_o, eo
    assert es < TOL_STATE, es
    assert en < TOL_STATE, en
    # and per (sequence, head): outputs, final states and every valid snapshot
    wo = worst_seq_head(to_np(out), o_ref, c["cu_seqlens"])
    ws = worst_state(pool.cpu().numpy()[c["final_slot"]], s_ref)
    wn = worst_state(snap.cpu().numpy()[valid], snap_ref[valid]) if valid.any() else 0.0
    assert wo < tol_o, wo
    assert ws < TOL_STATE, ws
    assert wn < TOL_STATE, wn
    return eo, es, en


def test_many_chunks_several_heads(kda):
    c = W.prefill_case(50, [1000, 64, 333, 1], 4, pool_slots=8, track_per_seq=3)
    check(c, run(kda, c))


def test_longest_first_schedule_gives_identical_results(kda):
    c = W.prefill_case(51, [90, 700, 5, 300], 2, pool_slots=6, track_per_seq=2)
    a = run(kda, c)
    b = run(kda, c, workspace=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_fp32_output_from_bf16_inputs(kda):
    c = W.prefill_case(52, [200, 77], 2, pool_slots=4)
    check(c, run(kda, c, out_dtype=torch.float32), tol_o=TOL_STATE)


@pytest.mark.parametrize("flags", [1, 2, 3])
def test_preactivated_gate_and_beta_flags(kda, flags):
    c = W.prefill_case(53, [150, 64], 2, pool_slots=4)
    if flags & 1:  # gate input holds g = log decay (<= 0)
        g = -np.abs(W.bf16_bits_to_f32(c["gate"])) * 0.5
        c["gate"] = W.f32_to_bf16_bits(g)
    if flags & 2:  # beta input holds beta in (0, 1)
        b = 1.0 / (1.0 + np.exp(-W.bf16_bits_to_f32(c["beta"])))
        c["beta"] = W.f32_to_bf16_bits(b.astype(np.float32))
    check(c, run(kda, c, flags=flags), flags=flags)


def test_strong_decay_chunks_use_the_exact_fallback(kda):
    # raw gates of +30 make 1/alpha = 1 + e^30 per token: a half chunk's factor
    # passes 2^64 after two such tokens, so those chunks take the token path
    c = W.prefill_case(54, [256, 100], 2, pool_slots=4, track_per_seq=2)
    g = W.bf16_bits_to_f32(c["gate"]).copy()
    g[10:14] = 30.0        # chunk 0 of sequence 0
    g[200:203, 1] = 45.0   # chunk 3 of sequence 0, head 1 only
    c["gate"] = W.f32_to_bf16_bits(g)
    check(c, run(kda, c))


def test_chunk_vs_recurrent_gap_is_reported(kda, capsys):
    c = W.prefill_case(55, [2048, 700], 4, pool_slots=4, track_per_seq=2)
    a = run(kda, c)
    b = run(kda, c, flags=kda.KDA_PREFILL_RECURRENT)
    gc = check(c, a)
    gr = check(c, b)
    gap_o = rel_l2(to_np(a[0]), to_np(b[0]))
    gap_s = rel_l2(a[1].cpu().numpy(), b[1].cpu().numpy())
    with capsys.disabled():
        print(f"\n[chunk vs recurrent] vs oracle (out, state, snapshot): chunk {gc}, "
              f"recurrent {gr}; chunk-recurrent gap: out {gap_o:.3e}, state {gap_s:.3e}")
    assert gap_s < 2 * TOL_STATE
