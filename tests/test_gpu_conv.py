"""GPU parity of kda_conv_compact (byte copy: bit-exact against the oracle),
alone and chained after the fused accept + commit on the same stream."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import i32

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


def _dev(pool, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(pool).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(pool)).cuda()


def _host(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16) if dtype == "bf16" else a


@pytest.mark.parametrize("keep", [1, 3, 5, 8])
@pytest.mark.parametrize("channels,dtype", [(4096, "bf16"), (200, "bf16"), (100, "f32")])
def test_conv_compact_bit_exact(kda, keep, channels, dtype):
    """37 requests, three tensors; 4096 bf16 channels span two CTAs per row,
    200 and 100 channels leave a ragged last chunk."""
    c = W.conv_case(300 + keep, 37, 7, keep, channels, 3, 50, dtype=dtype)
    slots = c["slots"].copy()
    slots[5] = -1  # padding request
    pools = [_dev(p, dtype) for p in c["pools"]]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_conv_compact(pools, i32(slots), i32(c["num_accepted"]), keep, dev_status=st)
    torch.cuda.synchronize()
    want, st_ref = oracle.conv_compact(c["pools"], slots, c["num_accepted"], keep)
    assert int(st.item()) == st_ref == 0
    for got, w in zip(pools, want):
        assert np.array_equal(_host(got, dtype), w)


def test_conv_compact_bad_inputs_and_mixed_tensors(kda):
    keep, K = 3, 4
    c = W.conv_case(310, 6, K, keep, 64, 1, 8, dtype="f32")
    big = W.conv_case(311, 6, K, keep, 2048, 1, 8, dtype="bf16")
    slots = c["slots"].copy()
    acc = c["num_accepted"].copy()
    slots[0] = 8           # past the pool: BAD_SLOT
    acc[1] = K + 1         # a + keep > rows: BAD_ACCEPT
    acc[2] = -1            # BAD_ACCEPT
    acc[3] = 0             # unchanged
    pools = [_dev(c["pools"][0], "f32"), _dev(big["pools"][0], "bf16")]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_conv_compact(pools, i32(slots), i32(acc), keep, dev_status=st)
    torch.cuda.synchronize()
    want, st_ref = oracle.conv_compact([c["pools"][0], big["pools"][0]], slots, acc, keep)
    assert int(st.item()) == st_ref == (kda.KDA_DEV_BAD_SLOT | kda.KDA_DEV_BAD_ACCEPT)
    assert np.array_equal(_host(pools[0], "f32"), want[0])
    assert np.array_equal(_host(pools[1], "bf16"), want[1])


def test_accept_commit_then_conv_compact(kda):
    """The post-sampling step on one stream: accepted lengths from token ids,
    the recurrent-state rebuild, then the conv windows of q, k and v; draftless
    requests (q_len = 1) shift their windows by one."""
    R, K, H, keep = 12, 7, 2, 3
    ql = np.array([7, 1, 7, 3, 1, 5, 7, 2, 7, 4, 6, 1], np.int32)
    s = W.spec_case(320, R, K, H, P=16, q_len=ql)
    a = W.accept_case(321, R, K, q_len=ql, p_match=0.7)
    c = W.conv_case(322, R, K, keep, 4096, 3, 16, dtype="bf16")
    convs = [_dev(p, "bf16") for p in c["pools"]]
    pool = torch.from_numpy(s["pool"]).cuda()
    rec_u = torch.randn(R, H, K, 128, device="cuda") * 0.1
    rec_kg = torch.randn(R, H, K, 256, device="cuda").to(torch.bfloat16)
    acc = torch.empty(R, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        kda.kda_spec_accept_commit(pool, i32(s["ckpt"]), i32(a["tokens"]), i32(a["sampled"]),
                                   rec_u, rec_kg, q_len=i32(ql), num_accepted=acc,
                                   dev_status=st, stream=stream)
        kda.kda_conv_compact(convs, i32(c["slots"]), acc, keep, dev_status=st, stream=stream)
    stream.synchronize()
    assert int(st.item()) == 0
    a_ref, _, _ = oracle.accept(a["tokens"], a["sampled"], K, q_len=ql)
    assert np.array_equal(acc.cpu().numpy(), a_ref)
    assert (a_ref[ql == 1] == 1).all()
    want, _ = oracle.conv_compact(c["pools"], c["slots"], a_ref, keep)
    for got, w in zip(convs, want):
        assert np.array_equal(_host(got, "bf16"), w)


@pytest.mark.parametrize("keep", [3, 9])
def test_fused_conv_windows_match_separate_launch(kda, keep):
    """kda_spec_accept_commit with conv tensors leaves the recurrent pool, the
    accepted lengths and every conv window bit-identical to the fused commit
    without them followed by kda_conv_compact; bad q_len and conv slots past
    the tensor are flagged the same way."""
    R, K, H = 20, 7, 2
    ql = np.random.default_rng(330).integers(1, K + 1, size=R).astype(np.int32)
    ql[3] = K + 3                                        # bad q_len: a = -1
    s = W.spec_case(331, R, K, H, P=24, q_len=np.clip(ql, 0, K))
    a = W.accept_case(332, R, K, q_len=np.clip(ql, 0, K), p_match=0.6)
    c4k = W.conv_case(333, R, K, keep, 4096, 2, 24, dtype="bf16")
    c100 = W.conv_case(334, R, K, keep, 100, 1, 24, dtype="f32")
    conv_slot = c4k["slots"].copy()
    conv_slot[7] = 30                                    # past every conv tensor
    conv_slot[8] = -1                                    # padding
    rec_u = torch.randn(R, H, K, 128, device="cuda") * 0.1
    rec_kg = torch.randn(R, H, K, 256, device="cuda").to(torch.bfloat16)
    res = []
    for fused in (False, True):
        pool = torch.from_numpy(s["pool"]).cuda()
        convs = [_dev(p, "bf16") for p in c4k["pools"]] + [_dev(c100["pools"][0], "f32")]
        acc = torch.empty(R, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kw = dict(q_len=i32(ql), num_accepted=acc, dev_status=st)
        if fused:
            kda.kda_spec_accept_commit(pool, i32(s["ckpt"]), i32(a["tokens"]), i32(a["sampled"]),
                                       rec_u, rec_kg, convs=convs, conv_slot=i32(conv_slot),
                                       conv_keep=keep, **kw)
        else:
            kda.kda_spec_accept_commit(pool, i32(s["ckpt"]), i32(a["tokens"]), i32(a["sampled"]),
                                       rec_u, rec_kg, **kw)
            kda.kda_conv_compact(convs, i32(conv_slot), acc, keep, dev_status=st)
        torch.cuda.synchronize()
        res.append((pool.cpu(), acc.cpu(), [x.cpu() for x in convs], int(st.item())))
    (p0, a0, c0, s0), (p1, a1, c1, s1) = res
    assert torch.equal(p0, p1) and torch.equal(a0, a1) and s0 == s1
    assert s1 == kda.KDA_DEV_BAD_ACCEPT | kda.KDA_DEV_BAD_SLOT
    for x, y in zip(c0, c1):
        assert torch.equal(x, y)
    a_ref, _, _ = oracle.accept(a["tokens"], a["sampled"], K, q_len=ql)
    want, _ = oracle.conv_compact(c4k["pools"] + c100["pools"], conv_slot, a_ref, keep)
    got = [x.numpy().view(np.uint16) for x in c1[:2]] + [c1[2].numpy()]
    for g, w in zip(got, want):
        assert np.array_equal(g, w)
