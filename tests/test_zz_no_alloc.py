"""kda_slot_copy_noalloc: the slot copy for callers that cannot allocate device
memory on demand (an engine whose pool allocator owns all device memory after
start-up, or a path where cudaMalloc and the device synchronisation it may
cause are not acceptable).  It keeps its scratch in a fixed array inside the
library and must give exactly what kda_slot_copy gives with a caller-provided
workspace, and what the oracle's slot copy gives, call after call.

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W

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


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _noalloc(kda, pool, sc):
    """Call the allocation-free entry point through the C ABI."""
    desc = (kda.PoolDesc * 1)()
    desc[0] = kda.PoolDesc(pool.data_ptr(), pool.stride(0) * pool.element_size(),
                           pool[0].numel() * pool.element_size(), pool.shape[0])
    clear, src, offs, dst = (_i32(sc[n]) for n in ("clear", "src", "dst_offsets", "dst"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = kda.lib().kda_slot_copy_noalloc(desc, 1, clear.data_ptr(), clear.numel(),
                                         src.data_ptr(), offs.data_ptr(), dst.data_ptr(),
                                         src.numel(), dst.numel(), status.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, int(status.item())


def _with_workspace(kda, pool, sc):
    ws = torch.empty(kda.kda_slot_copy_workspace_size(pool.shape[0]), dtype=torch.uint8,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_slot_copy([pool], _i32(sc["clear"]), _i32(sc["src"]), _i32(sc["dst_offsets"]),
                      _i32(sc["dst"]), ws, dev_status=status)
    torch.cuda.synchronize()
    return int(status.item())


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(kda):
    g = torch.Generator().manual_seed(7)
    base = torch.randn(300, 2, 128, 128, generator=g).cuda()
    first = W.slot_copy_case(61, 300, 6, 4, 9)
    # the second call reads slots the first one wrote: stale scratch from the
    # first call would flag a false overlap here
    second = W.slot_copy_case(62, 300, 5, 3, 4)
    free = np.setdiff1d(np.arange(300), np.concatenate([first["dst"], first["clear"]]))
    second["src"] = first["dst"][:5].astype(np.int32)
    rest = np.setdiff1d(free, second["src"])
    second["dst"] = rest[:15].astype(np.int32)
    second["clear"] = rest[15:19].astype(np.int32)
    a = base.clone()
    b = base.clone()
    for sc in (first, second):
        before = b.cpu().numpy()
        assert _with_workspace(kda, a, sc) == 0
        st, dev = _noalloc(kda, b, sc)
        assert st == 0 and dev == 0
        assert torch.equal(a, b)  # copies are exact: the tolerance is zero
        (want,) = oracle.slot_copy([before], sc["clear"], sc["src"], sc["dst_offsets"], sc["dst"])
        assert np.array_equal(b.cpu().numpy(), want)


def test_noalloc_still_detects_overlap(kda):
    pool = torch.randn(40, 64, device="cuda")
    before = pool.clone()
    sc = W.slot_copy_case(63, 40, 3, 2, 2)
    sc["dst"][1] = sc["dst"][0]
    st, dev = _noalloc(kda, pool, sc)
    assert st == 0 and dev & kda.KDA_DEV_OVERLAP
    assert torch.equal(pool, before)
    # and the next valid call is unaffected
    sc = W.slot_copy_case(64, 40, 3, 2, 2)
    ref = pool.clone()
    assert _with_workspace(kda, ref, sc) == 0
    st, dev = _noalloc(kda, pool, sc)
    assert st == 0 and dev == 0 and torch.equal(pool, ref)


def test_noalloc_rejects_pools_beyond_its_fixed_size(kda):
    max_slots = 1 << 20
    desc = (kda.PoolDesc * 1)()
    desc[0] = kda.PoolDesc(1 << 20, 16, 16, max_slots + 1)  # never dereferenced
    offs = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = kda.lib().kda_slot_copy_noalloc(desc, 1, None, 0, None, offs.data_ptr(), None, 0, 0,
                                         None, None)
    assert st == 2  # KDA_ERR_UNSUPPORTED, nothing launched
    assert isinstance(ctypes.c_int(st).value, int)
