"""Failure detection without a GPU fault: a bounded in-kernel wait on a barrier
that nothing arrives on gives up, the status reaches the host, and the context
stays usable (the next launches run and are correct)."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import dev_tensor, i32, rel_l2, to_np, wid

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


def test_bounded_wait_gives_up_and_the_context_stays_usable(kda):
    st = torch.zeros(4, dtype=torch.int32, device="cuda")[:1]
    cycles = torch.zeros(2, dtype=torch.int64, device="cuda")[:1]
    kda.kda_selftest_bounded_wait(4096, st, cycles)
    torch.cuda.synchronize()
    assert int(st.item()) == kda.KDA_DEV_TIMEOUT
    per_poll = int(cycles.item()) / 4096
    assert per_poll > 0
    print(f"[bounded wait] {per_poll:.0f} cycles per poll; the kernels' 2^18 polls give up after "
          f"about {per_poll * (1 << 18) / 2.0e9:.2f} s at 2 GHz")
    # the same context runs a decode step correctly afterwards
    d = W.decode_case(500, 8, 2, 12)
    pool = torch.from_numpy(d["pool"]).cuda()
    out = torch.empty(8, 2, 128, dtype=torch.bfloat16, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_recurrent_decode(*(dev_tensor(d[n], "bf16") for n in ("q", "k", "v", "beta", "gate")),
                             pool, i32(d["slot"]), out, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    o_ref, p_ref, _ = oracle.decode(wid(d, "q"), wid(d, "k"), wid(d, "v"), wid(d, "beta"),
                                    wid(d, "gate"), d["pool"], d["slot"])
    assert rel_l2(to_np(out), o_ref) < 5e-3
    assert rel_l2(pool.cpu().numpy(), p_ref) < 1e-4
