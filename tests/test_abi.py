"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad host-side arguments before launching anything."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "kda.h"


@pytest.fixture(scope="module")
def kda():
    import __graft_entry__

    __graft_entry__.build()
    import serving_kda_chunk_gb300 as kda

    return kda


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("kda_chunk_prefill", "kda_recurrent_decode", "kda_spec_verify", "kda_spec_accept",
              "kda_spec_commit", "kda_spec_accept_commit", "kda_conv_compact", "kda_slot_copy"):
        assert f in names


def test_library_exports_every_declared_symbol(kda):
    L = ctypes.CDLL(str(kda.LIB_PATH))
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(kda):
    assert kda.kda_status_string(0) == "KDA_OK"
    assert "INVALID_ARG" in kda.kda_status_string(1)
    assert "UNSUPPORTED" in kda.kda_status_string(2)
    assert kda.kda_abi_version() >= 104


def test_prefill_workspace_size(kda):
    # every (chunk, head)'s operand block (132 096 bytes), one fp32 state per (sequence, head) for
    # the pipelined long-sequence path, for up to 8 sequences of on average at least 256 chunks
    # 48 more per (sequence, head) (the segment scan's start, Phi and B states, up to 16
    # segments), and a plan area well under 1 MiB
    H = 32
    for T, N in [(0, 1), (64, 1), (41460, 8), (255 * 64, 1), (256 * 64, 1), (131072, 1), (1 << 20, 8),
                 (1 << 20, 9), (2 * 256 * 64 - 200, 2)]:
        n_max = (T + 63 * N) // 64
        ws = kda.kda_chunk_prefill_workspace_size(T, N, H)
        scan = 48 * N * H * 128 * 128 * 4 if N <= 8 and n_max >= 256 * N else 0
        blocks = n_max * H * 132096 + N * H * 128 * 128 * 4 + scan
        assert ws % 16 == 0
        assert blocks <= ws < blocks + (1 << 20)
    assert kda.kda_chunk_prefill_workspace_size(1000, 2, 4) <= kda.kda_chunk_prefill_workspace_size(2000, 2, 4)


def test_workspace_sizes(kda):
    assert kda.kda_slot_copy_workspace_size(0) == 16
    assert kda.kda_slot_copy_workspace_size(4096) == 16 + 4096 // 8
    assert kda.kda_slot_copy_workspace_size(129) % 16 == 0
    assert kda.kda_chunk_prefill_workspace_size(1 << 20, 8, 32) >= 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced (checks fail first)


def test_host_checks_reject_bad_arguments(kda):
    L = kda.lib()
    # unsupported head dimension
    st = L.kda_recurrent_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 2, 64, 64, 1.0, 0, FAKE, 8,
                                FAKE, FAKE, 0, None, None)
    assert st == 2
    # null input pointer
    st = L.kda_recurrent_decode(None, FAKE, FAKE, FAKE, FAKE, 0, 4, 2, 128, 128, 1.0, 0, FAKE, 8,
                                FAKE, FAKE, 0, None, None)
    assert st == 1
    # misaligned output
    st = L.kda_recurrent_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 2, 128, 128, 1.0, 0, FAKE, 8,
                                FAKE, FAKE + 2, 0, None, None)
    assert st == 1
    # bad dtype enum
    st = L.kda_spec_verify(FAKE, FAKE, FAKE, FAKE, FAKE, 7, 4, 3, None, 2, 128, 128, 1.0, 0, FAKE,
                           8, FAKE, FAKE, FAKE, FAKE, 0, None, None)
    assert st == 2
    # commit: K above the supported maximum
    st = L.kda_spec_commit(FAKE, 8, FAKE, None, FAKE, None, 4, 1000, 2, 128, 128, 0, FAKE, FAKE,
                           0, None, None, None)
    assert st == 2
    # accept: K = 0, K above one warp, null or misaligned pointers
    assert L.kda_spec_accept(FAKE, FAKE, None, 4, 0, FAKE, None, None, None) == 1
    assert L.kda_spec_accept(FAKE, FAKE, None, 4, 33, FAKE, None, None, None) == 2
    assert L.kda_spec_accept(FAKE, None, None, 4, 7, FAKE, None, None, None) == 1
    assert L.kda_spec_accept(FAKE, FAKE, FAKE + 4, 4, 7, FAKE, None, None, None) == 1
    assert L.kda_spec_accept(FAKE, FAKE, None, 4, 7, FAKE, FAKE + 8, None, None) == 1
    assert L.kda_spec_accept(None, None, None, 0, 7, None, None, None, None) == 0
    # fused accept + commit: missing sampled ids, K = 0, K above one warp
    args = lambda tok, smp, K: (FAKE, 8, FAKE, None, tok, smp, None, 4, K, 2, 128, 128, 0,  # noqa: E731
                                FAKE, FAKE, 0, None, None, None, None, None, None)
    assert L.kda_spec_accept_commit(*args(FAKE, None, 7)) == 1
    assert L.kda_spec_accept_commit(*args(FAKE, FAKE, 0)) == 1
    assert L.kda_spec_accept_commit(*args(FAKE, FAKE, 33)) == 2
    # fused conv windows: more than KDA_MAX_POOLS tensors, or no conv slots
    conv = (kda.ConvDesc * 1)()
    conv[0] = kda.ConvDesc(FAKE, 10 * 8192, 8192, 10, 8)
    a = list(args(FAKE, FAKE, 7))
    a[19] = ctypes.byref(kda.CommitExtras(conv, FAKE, None, None, None, 17, 3, 0, 0))
    assert L.kda_spec_accept_commit(*a) == 1
    a[19] = ctypes.byref(kda.CommitExtras(conv, None, None, None, None, 1, 3, 0, 0))
    assert L.kda_spec_accept_commit(*a) == 1
    # align mode: block size below K cannot hold one step's span; zero block size
    a[19] = ctypes.byref(kda.CommitExtras(conv, None, FAKE, FAKE, None, 0, 0, 6, 0))
    assert L.kda_spec_accept_commit(*a) == 2
    a[19] = ctypes.byref(kda.CommitExtras(conv, None, FAKE, FAKE, None, 0, 0, 0, 0))
    assert L.kda_spec_accept_commit(*a) == 1
    # prefill: chunk other than 64
    st = L.kda_chunk_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 64, 2, 128, 128, 32, 1.0,
                             0, None, 0, None, None, None, 0, None, FAKE, 0, None, 0, None, None)
    assert st == 2
    # prefill: snapshots requested without a snapshot buffer
    st = L.kda_chunk_prefill(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 1, 64, 2, 128, 128, 64, 1.0,
                             0, None, 0, None, None, FAKE, 1, None, FAKE, 0, None, 0, None, None)
    assert st == 1
    # both 16-bit state types at once
    both = kda.KDA_STATE_BF16 | kda.KDA_STATE_F16
    st = L.kda_recurrent_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 2, 128, 128, 1.0, both, FAKE,
                                8, FAKE, FAKE, 0, None, None)
    assert st == 2
    # zero-sized work launches nothing and succeeds
    assert L.kda_recurrent_decode(None, None, None, None, None, 0, 0, 2, 128, 128, 1.0, 0, None,
                                  0, None, None, 0, None, None) == 0


def test_slot_copy_host_checks(kda):
    L = kda.lib()
    descs = (kda.PoolDesc * 1)()
    descs[0] = kda.PoolDesc(FAKE, 64, 64, 8)
    # too many pools
    assert L.kda_slot_copy(descs, 17, None, 0, None, FAKE, None, 0, 0, FAKE, 4096, None,
                           None) == 1
    # slot_bytes not a multiple of 16
    descs[0] = kda.PoolDesc(FAKE, 64, 60, 8)
    assert L.kda_slot_copy(descs, 1, None, 0, None, FAKE, None, 0, 0, FAKE, 4096, None,
                           None) == 1
    # workspace too small
    descs[0] = kda.PoolDesc(FAKE, 64, 64, 1 << 20)
    assert L.kda_slot_copy(descs, 1, None, 0, None, FAKE, None, 0, 0, FAKE, 16, None,
                           None) == 1


def test_conv_compact_host_checks(kda):
    L = kda.lib()
    descs = (kda.ConvDesc * 2)()
    ok = kda.ConvDesc(FAKE, 10 * 8192, 8192, 10, 8)
    descs[0] = ok
    args = lambda n, keep: (descs, n, FAKE, FAKE, 4, keep, None, None)  # noqa: E731
    assert L.kda_conv_compact(*args(0, 3)) == 1            # no tensors
    assert L.kda_conv_compact(*args(17, 3)) == 1           # more than KDA_MAX_POOLS
    assert L.kda_conv_compact(*args(1, 0)) == 1            # keep 0
    assert L.kda_conv_compact(*args(1, 11)) == 1           # keep > rows
    descs[0] = kda.ConvDesc(FAKE + 8, 10 * 8192, 8192, 10, 8)
    assert L.kda_conv_compact(*args(1, 3)) == 1            # misaligned base
    descs[0] = kda.ConvDesc(FAKE, 10 * 8200, 8200, 10, 8)
    assert L.kda_conv_compact(*args(1, 3)) == 1            # row not a multiple of 16 bytes
    descs[0] = kda.ConvDesc(FAKE, 9 * 8192, 8192, 10, 8)
    assert L.kda_conv_compact(*args(1, 3)) == 1            # slots overlap
    descs[0] = ok
    assert L.kda_conv_compact(descs, 1, None, None, 0, 3, None, None) == 0  # nothing to do
    assert L.kda_conv_compact(descs, 1, None, FAKE, 4, 3, None, None) == 1  # null slots


def test_product_path_has_no_cpu_fallback():
    # the binding imports nothing from the oracle and no torch CPU op computes a result
    src = (ROOT / "serving_kda_chunk_gb300" / "__init__.py").read_text()
    assert "oracle" not in src.replace("no oracle", "")
    for f in (ROOT / "serving_kda_chunk_gb300" / "csrc").glob("*"):
        assert "oracle" not in f.read_text().lower(), f


def test_binding_rejects_mixed_activation_dtypes(kda):
    torch = pytest.importorskip("torch")
    q = torch.zeros(2, 1, 128, dtype=torch.bfloat16)
    k = torch.zeros(2, 1, 128, dtype=torch.float32)  # one tensor of another dtype
    beta = torch.zeros(2, 1, dtype=torch.bfloat16)
    pool = torch.zeros(1, 1, 128, 128)
    slot = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="one dtype"):
        kda.kda_recurrent_decode(q, k, q, beta, q, pool, slot, q)


def test_binding_rejects_index_tensors_that_are_not_int32(kda):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="int32"):
        kda._idx(torch.zeros(4, dtype=torch.int64), "slot")
    with pytest.raises(ValueError, match="fp32"):
        kda._f32(torch.zeros(4, dtype=torch.bfloat16), "rec_u")
    assert kda._idx(None, "slot") is None


def test_verify_binding_checks_rows_and_record_dtype(kda):
    torch = pytest.importorskip("torch")
    x = torch.zeros(10, 1, 128, dtype=torch.bfloat16)  # 10 rows: not R * K for K = 3
    beta = torch.zeros(10, 1, dtype=torch.bfloat16)
    pool = torch.zeros(1, 1, 128, 128)
    ckpt = torch.zeros(3, dtype=torch.int32)
    rec_u = torch.zeros(3, 1, 3, 128)
    with pytest.raises(ValueError, match="multiple of K"):
        kda.kda_spec_verify(x, x, x, beta, x, pool, ckpt, rec_u, x, x, K=3)
    x9, beta9 = x[:9], beta[:9]
    rec_kg = torch.zeros(3, 1, 3, 256)  # fp32 records for bf16 activations
    with pytest.raises(ValueError, match="rec_kg"):
        kda.kda_spec_verify(x9, x9, x9, beta9, x9, pool, ckpt, rec_u, rec_kg, x9, K=3)


def test_marshalling_matches_the_declared_signatures(kda, monkeypatch):
    """Every binding passes exactly the C signature's arguments, each convertible by its
    declared ctypes type (checked against a recording stand-in for the library, on CPU
    tensors, so no kernel runs)."""
    torch = pytest.importorskip("torch")
    real = kda.lib()
    calls = {}

    class Fake:
        def __getattr__(self, name):
            fn = getattr(real, name)

            def call(*args):
                assert len(args) == len(fn.argtypes), (name, len(args), len(fn.argtypes))
                for a, t in zip(args, fn.argtypes):
                    t.from_param(a)  # raises on a value the C type cannot take
                calls[name] = args
                return 0

            return call

    monkeypatch.setattr(kda, "_lib", Fake())
    monkeypatch.setattr(kda, "_p", lambda t: None if t is None else (
        t.data_ptr() if isinstance(t, torch.Tensor) else int(t)))
    monkeypatch.setattr(kda, "_p_any", lambda t: t.data_ptr())
    monkeypatch.setattr(kda, "_stream", lambda s: 0)
    bf, i32 = torch.bfloat16, torch.int32
    T, H, R, K = 128, 2, 3, 4
    x = torch.zeros(T, H, 128, dtype=bf)
    pool = torch.zeros(4, H, 128, 128)
    st = torch.zeros(1, dtype=i32)
    kda.kda_chunk_prefill(x, x, x, torch.zeros(T, H, dtype=bf), x,
                          torch.tensor([0, 64, 128], dtype=i32), x, state_pool=pool,
                          init_slot=torch.zeros(2, dtype=i32), final_slot=torch.ones(2, dtype=i32),
                          track_chunk_idx=torch.zeros(2, 1, dtype=i32),
                          track_state=torch.zeros(2, 1, H, 128, 128), dev_status=st)
    xd = torch.zeros(R, H, 128, dtype=bf)
    kda.kda_recurrent_decode(xd, xd, xd, torch.zeros(R, H, dtype=bf), xd, pool,
                             torch.zeros(R, dtype=i32), xd, dev_status=st)
    xs = torch.zeros(R * K, H, 128, dtype=bf)
    rec_u = torch.zeros(R, H, K, 128)
    rec_kg = torch.zeros(R, H, K, 256, dtype=bf)
    idx = torch.zeros(R, dtype=i32)
    kda.kda_spec_verify(xs, xs, xs, torch.zeros(R * K, H, dtype=bf), xs, pool, idx, rec_u, rec_kg,
                        xs, K=K, q_len=idx, dev_status=st)
    tok = torch.zeros(R, K, dtype=i32)
    kda.kda_spec_accept(tok, tok, idx, q_len=idx, next_token=idx, dev_status=st)
    kda.kda_spec_commit(pool, idx, idx, rec_u, rec_kg, K=K, dst_slot=idx, q_len=idx,
                        plan_out=torch.zeros(R, 3, dtype=i32), dev_status=st)
    conv = torch.zeros(4, 6, 64, dtype=bf)
    kda.kda_spec_accept_commit(pool, idx, tok, tok, rec_u, rec_kg, dst_slot=idx, q_len=idx,
                               num_accepted=idx, next_token=idx, convs=[conv, conv],
                               conv_slot=idx, conv_keep=2, seq_len0=idx, block_size=16,
                               block_slot=idx, block_idx_out=idx, dev_status=st)
    kda.kda_conv_compact([conv], idx, idx, 2, dev_status=st)
    sets = (torch.zeros(1, dtype=i32), torch.zeros(1, dtype=i32), torch.tensor([0, 1], dtype=i32),
            torch.ones(1, dtype=i32))
    kda.kda_slot_copy([pool], *sets, torch.zeros(64, dtype=torch.uint8), dev_status=st)
    kda.kda_slot_copy_noalloc([pool], *sets, dev_status=st)
    kda.kda_selftest_bounded_wait(8, st)
    assert set(calls) == {"kda_chunk_prefill", "kda_recurrent_decode", "kda_spec_verify",
                          "kda_spec_accept", "kda_spec_commit", "kda_spec_accept_commit",
                          "kda_conv_compact", "kda_slot_copy", "kda_slot_copy_noalloc",
                          "kda_selftest_bounded_wait"}
    # a few positions that matter: sizes and the state-type flag bits
    assert calls["kda_spec_verify"][6:8] == (R, K)
    assert calls["kda_spec_commit"][6:9] == (R, K, H)
    assert calls["kda_slot_copy"][7:9] == (1, 1)


def _have(tool):
    import shutil

    return shutil.which(tool) is not None


@pytest.mark.skipif(not (_have("gcc") and _have("g++")), reason="needs gcc and g++")
def test_header_is_standalone_c_and_cxx(tmp_path):
    import subprocess

    src = tmp_path / "use.c"
    src.write_text('#include "kda.h"\nint main(void) { return 0; }\n')
    inc = f"-I{ROOT / 'include'}"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", inc,
                    "-fsyntax-only", str(src)], check=True)
    cxx = tmp_path / "use.cpp"
    cxx.write_text(src.read_text())
    subprocess.run(["g++", "-std=c++11", "-Wall", "-Wextra", "-pedantic", "-Werror", inc,
                    "-fsyntax-only", str(cxx)], check=True)


@pytest.mark.skipif(not _have("gcc"), reason="needs gcc")
def test_plain_c_caller_links_and_gets_host_errors(kda, tmp_path):
    """A C program built against the header and the shared library alone: it gets
    the version and status strings, and host-checkable errors come back as status
    codes before anything reaches a GPU."""
    import subprocess

    src = tmp_path / "caller.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "kda.h"
int main(void) {
    if (kda_abi_version() < 104) return 1;
    if (strcmp(kda_status_string(KDA_OK), "KDA_OK") != 0) return 2;
    /* d_k != 128 is unsupported: refused on the host, nothing launched */
    kda_status s = kda_recurrent_decode(0, 0, 0, 0, 0, KDA_BF16, 1, 1, 64, 128, 1.0f, 0u,
                                        0, 1, 0, 0, KDA_BF16, 0, 0);
    if (s != KDA_ERR_UNSUPPORTED) return 3;
    /* R = 0 launches nothing and succeeds */
    if (kda_spec_accept(0, 0, 0, 0, 4, 0, 0, 0, 0) != KDA_OK) return 4;
    puts("ok");
    return 0;
}
''')
    exe = tmp_path / "caller"
    libdir = str(Path(kda.LIB_PATH).parent)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{ROOT / 'include'}", str(src),
                    f"-L{libdir}", "-lkda", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stderr)
