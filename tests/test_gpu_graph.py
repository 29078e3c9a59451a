"""The serving step captured in one CUDA graph: every entry point is
asynchronous, allocates nothing and never synchronises with the host, so a
decode + verify + fused accept/commit (+ conv windows) + slot copy sequence
captures as is, and its replay leaves the same bits as the eager calls."""
import numpy as np
import pytest

import workloads as W
from helpers import dev_tensor, i32

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


def _step_buffers(kda):
    R, K, H = 16, 7, 4
    d = W.decode_case(400, 24, H, 40)
    s = W.spec_case(401, R, K, H, P=R)
    a = W.accept_case(402, R, K, p_match=0.7)
    c = W.conv_case(403, R, K, 3, 512, 2, R, dtype="bf16")
    sc = W.slot_copy_case(404, 32, 3, 2, 4)
    bufs = dict(
        dec=[dev_tensor(d[n], "bf16") for n in ("q", "k", "v", "beta", "gate")],
        dpool=torch.from_numpy(d["pool"]).cuda(), dslot=i32(d["slot"]),
        dout=torch.empty(24, H, 128, dtype=torch.bfloat16, device="cuda"),
        spec=[dev_tensor(s[n], "bf16") for n in ("q", "k", "v", "beta", "gate")],
        spool=torch.from_numpy(s["pool"]).cuda(), ckpt=i32(s["ckpt"]),
        rec_u=torch.empty(R, H, K, 128, device="cuda"),
        rec_kg=torch.empty(R, H, K, 256, dtype=torch.bfloat16, device="cuda"),
        sout=torch.empty(R * K, H, 128, dtype=torch.bfloat16, device="cuda"),
        tok=i32(a["tokens"]), smp=i32(a["sampled"]),
        acc=torch.empty(R, dtype=torch.int32, device="cuda"),
        convs=[torch.from_numpy(x.view(np.int16)).cuda() for x in c["pools"]],
        cslot=i32(c["slots"]),
        cpool=torch.randn(32, H, 128, 128, device="cuda"),
        sc={n: i32(sc[n]) for n in ("clear", "src", "dst_offsets", "dst")},
        ws=torch.empty(kda.kda_slot_copy_workspace_size(32), dtype=torch.uint8, device="cuda"),
        st=torch.zeros(1, dtype=torch.int32, device="cuda"),
        K=K)
    return bufs


def _run_step(kda, b, stream):
    kda.kda_recurrent_decode(*b["dec"], b["dpool"], b["dslot"], b["dout"], dev_status=b["st"],
                             stream=stream)
    kda.kda_spec_verify(*b["spec"], b["spool"], b["ckpt"], b["rec_u"], b["rec_kg"], b["sout"],
                        K=b["K"], dev_status=b["st"], stream=stream)
    kda.kda_spec_accept_commit(b["spool"], b["ckpt"], b["tok"], b["smp"], b["rec_u"], b["rec_kg"],
                               num_accepted=b["acc"], convs=b["convs"], conv_slot=b["cslot"],
                               conv_keep=3, dev_status=b["st"], stream=stream)
    sc = b["sc"]
    kda.kda_slot_copy([b["cpool"]], sc["clear"], sc["src"], sc["dst_offsets"], sc["dst"], b["ws"],
                      dev_status=b["st"], stream=stream)


def test_serving_step_replays_in_a_cuda_graph(kda):
    eager = _step_buffers(kda)
    graphed = _step_buffers(kda)
    torch.manual_seed(7)
    init = graphed["cpool"].clone()
    eager["cpool"].copy_(init)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    # capture records the launches without running them; the buffers still hold the inputs
    with torch.cuda.graph(g, stream=stream):
        _run_step(kda, graphed, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for _ in range(2):  # two steps: the second one starts from the first one's states
        g.replay()
        with torch.cuda.stream(stream):
            _run_step(kda, eager, stream)
    torch.cuda.synchronize()
    assert int(eager["st"].item()) == 0 and int(graphed["st"].item()) == 0
    for name in ("dout", "dpool", "sout", "rec_u", "rec_kg", "spool", "acc", "cpool"):
        assert torch.equal(eager[name], graphed[name]), name
    for x, y in zip(eager["convs"], graphed["convs"]):
        assert torch.equal(x, y)


@pytest.mark.parametrize("shape", ["batched", "one_long_sequence", "one_long_sequence_32_heads"])
def test_two_phase_prefill_replays_in_a_cuda_graph(kda, shape):
    # the plan / prep / sweep launches (for one long sequence with 2 heads the segment scan's
    # launches and its combine, with 32 heads the pipelined segment launches) capture as they
    # are; two replays match two eager calls bit for bit
    lengths = [300, 65, 1] if shape == "batched" else [256 * 64 + 3]
    H = 32 if shape == "one_long_sequence_32_heads" else 2
    c = W.prefill_case(405, lengths, H, pool_slots=4, track_per_seq=2)
    N, H, T = c["N"], c["H"], c["T"]
    M = c["track"].shape[1]
    tok = [dev_tensor(c[n], "bf16") for n in ("q", "k", "v", "beta", "gate")]
    idx = dict(cu=i32(c["cu_seqlens"]), init=i32(c["init_slot"]), fin=i32(c["final_slot"]),
               track=i32(c["track"]))

    def buffers():
        return dict(pool=torch.from_numpy(c["pool"]).cuda(),
                    out=torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda"),
                    snap=torch.zeros(N, M, H, 128, 128, device="cuda"),
                    ws=torch.empty(kda.kda_chunk_prefill_workspace_size(T, N, H), dtype=torch.uint8,
                                   device="cuda"),
                    st=torch.zeros(1, dtype=torch.int32, device="cuda"))

    def call(b, stream):
        kda.kda_chunk_prefill(*tok, idx["cu"], b["out"], state_pool=b["pool"], init_slot=idx["init"],
                              final_slot=idx["fin"], track_chunk_idx=idx["track"], track_state=b["snap"],
                              workspace=b["ws"], dev_status=b["st"], stream=stream)

    eager, graphed = buffers(), buffers()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call(graphed, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for _ in range(2):  # in place: the second call starts from the first one's final states
        g.replay()
        with torch.cuda.stream(stream):
            call(eager, stream)
    torch.cuda.synchronize()
    assert int(eager["st"].item()) == 0 and int(graphed["st"].item()) == 0
    for name in ("pool", "out", "snap"):
        assert torch.equal(eager[name], graphed[name]), name
