"""One activation code path: the same raw gate gives the same decay bits in
every entry point ("state semantics" page, section 4: where the gate is
activated is a replay-consistency hazard between prefill, decode and verify).

With raw beta = -inf (beta = 0 exactly) every path reduces one token to
S_1 = Diag(alpha) S_0: u = 0, so the key write adds exact zeros and each state
element is alpha_i * S_0 rounded once.  The final states of decode, of verify
followed by a one-position commit, of the tensor-core prefill and of the
token-serial prefill must then agree bit for bit; any difference in how a
kernel turns the raw gate into alpha shows up in the last bit."""
import numpy as np
import pytest

import workloads as W
from helpers import TOL_STATE, dev_tensor, i32, rel_l2

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


NEG_INF_BF16 = np.uint16(0xFF80)


def _case(seed, R, H):
    c = W.decode_case(seed, R, H, R)
    c["beta"] = np.full_like(c["beta"], NEG_INF_BF16)
    # spread raw gates over strong and weak decays, plus exact edges
    rng = np.random.default_rng(seed + 1000)
    g = (rng.standard_normal(c["gate"].shape, dtype=np.float32) * 4.0).astype(np.float32)
    g[0, 0, :4] = [-np.inf, 0.0, -30.0, 30.0]
    c["gate"] = W.f32_to_bf16_bits(g)
    return c


def test_gate_decay_bits_agree_across_entry_points(kda):
    R, H = 8, 4
    c = _case(7, R, H)
    slots = np.arange(R, dtype=np.int32)
    tok = {n: dev_tensor(c[n], "bf16") for n in ("q", "k", "v", "beta", "gate")}
    S0 = torch.from_numpy(c["pool"][slots]).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    # decode: one step in place
    p_dec = S0.clone()
    out = torch.empty(R, H, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_recurrent_decode(tok["q"], tok["k"], tok["v"], tok["beta"], tok["gate"], p_dec,
                             i32(slots), out, dev_status=st)

    # verify (K = 1) then commit a = 1 from the records
    p_spec = S0.clone()
    rec_u = torch.empty(R, H, 1, 128, device="cuda")
    rec_kg = torch.empty(R, H, 1, 256, dtype=torch.bfloat16, device="cuda")
    sout = torch.empty(R, H, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_spec_verify(tok["q"], tok["k"], tok["v"], tok["beta"], tok["gate"], p_spec,
                        i32(slots), rec_u, rec_kg, sout, K=1, dev_status=st)
    kda.kda_spec_commit(p_spec, i32(slots), i32(np.ones(R, np.int32)), rec_u, rec_kg, K=1,
                        dev_status=st)

    # prefill: every request as a one-token sequence from its slot, final state in place
    cu = i32(np.arange(R + 1, dtype=np.int32))
    pre = {}
    for name, flags in (("tc", 0), ("serial", kda.KDA_PREFILL_RECURRENT)):
        p = S0.clone()
        o = torch.empty(R, H, 128, dtype=torch.bfloat16, device="cuda")
        kda.kda_chunk_prefill(tok["q"], tok["k"], tok["v"], tok["beta"], tok["gate"], cu, o,
                              state_pool=p, init_slot=i32(slots), final_slot=i32(slots),
                              flags=flags, dev_status=st)
        pre[name] = p
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.all(rec_u == 0)  # beta = 0: no correction
    ref = p_dec.cpu().numpy()
    for name, p in (("verify+commit", p_spec), ("tc prefill", pre["tc"]),
                    ("serial prefill", pre["serial"])):
        got = p.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), name
    # and the decay itself is the definition's, alpha = 1 / (1 + e^x) per key channel
    x = W.widen(c["gate"], "bf16")
    alpha = 1.0 / (1.0 + np.exp(x))
    want = c["pool"][slots].astype(np.float64) * alpha[:, :, None, :]
    assert rel_l2(ref, want) < TOL_STATE
    # raw -inf is alpha = 1 exactly: that key channel is copied unchanged
    assert np.array_equal(ref[0, 0, :, 0], c["pool"][0, 0, :, 0])
