"""Python binding of libkda, the sm_103a library for the KDA recurrent-state path.

Argument marshalling only: every function below turns torch tensors into
device pointers and sizes and calls the C ABI declared in include/kda.h; all
arithmetic runs in the library's CUDA kernels.  There is no CPU fallback: if
libkda.so is missing the import of the library raises.

Entry points (same names as the C ABI):
  kda_chunk_prefill, kda_recurrent_decode, kda_spec_verify, kda_spec_accept, kda_spec_commit,
  kda_spec_accept_commit, kda_conv_compact, kda_slot_copy, kda_slot_copy_noalloc,
  kda_chunk_prefill_workspace_size, kda_slot_copy_workspace_size.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

__all__ = [
    "KDA_BF16", "KDA_F32", "KDA_GATE_LOG", "KDA_BETA_ACT", "KDA_STATE_BF16", "KDA_STATE_F16",
    "KDA_QK_L2NORM",
    "KdaError", "lib",
    "kda_chunk_prefill", "kda_recurrent_decode", "kda_spec_verify", "kda_spec_accept",
    "kda_spec_commit", "kda_spec_accept_commit", "kda_conv_compact", "kda_slot_copy",
    "kda_slot_copy_noalloc", "kda_chunk_prefill_workspace_size",
    "kda_slot_copy_workspace_size",
    "kda_status_string", "kda_abi_version", "kda_selftest_bounded_wait", "PoolDesc",
    "ConvDesc", "CommitExtras",
]

KDA_BF16, KDA_F32 = 0, 1
KDA_GATE_LOG, KDA_BETA_ACT, KDA_PREFILL_RECURRENT = 1, 2, 4
KDA_STATE_BF16, KDA_STATE_F16 = 8, 16
KDA_QK_L2NORM = 32
KDA_DEV_BAD_SLOT, KDA_DEV_BAD_TRACK, KDA_DEV_BAD_ACCEPT = 1, 2, 4
KDA_DEV_BAD_SEQLEN, KDA_DEV_OVERLAP, KDA_DEV_TIMEOUT = 8, 16, 32
KDA_MAX_POOLS = 16

LIB_PATH = Path(__file__).resolve().parent / "libkda.so"
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {kda_status_string(status)} (status {status})")
        self.status = status


class PoolDesc(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("slot_stride_bytes", ctypes.c_int64),
                ("slot_bytes", ctypes.c_int64), ("num_slots", ctypes.c_int64)]


class ConvDesc(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("slot_stride_bytes", ctypes.c_int64),
                ("row_bytes", ctypes.c_int64), ("n_rows", ctypes.c_int32),
                ("num_slots", ctypes.c_int32)]


class CommitExtras(ctypes.Structure):
    _fields_ = [("convs", ctypes.POINTER(ConvDesc)), ("conv_slot", ctypes.c_void_p),
                ("seq_len0", ctypes.c_void_p), ("block_slot", ctypes.c_void_p),
                ("block_idx_out", ctypes.c_void_p), ("n_convs", ctypes.c_int32),
                ("conv_keep", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


def lib():
    """The loaded C library with argument types set (raises if not built)."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback path)")
        L = ctypes.CDLL(str(LIB_PATH))
        vp, i32, i64, f32, u32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                      ctypes.c_float, ctypes.c_uint32, ctypes.c_size_t)
        L.kda_chunk_prefill.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, vp, i32, i32, i32, i32,
                                        i32, i32, f32, u32, vp, i64, vp, vp, vp, i32, vp, vp,
                                        ctypes.c_int, vp, sz, vp, vp]
        L.kda_recurrent_decode.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, i32, i32, i32, i32,
                                           f32, u32, vp, i64, vp, vp, ctypes.c_int, vp, vp]
        L.kda_spec_verify.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, i32, i32, vp, i32, i32,
                                      i32, f32, u32, vp, i64, vp, vp, vp, vp, ctypes.c_int, vp, vp]
        L.kda_spec_commit.argtypes = [vp, i64, vp, vp, vp, vp, i32, i32, i32, i32, i32, u32, vp,
                                      vp, ctypes.c_int, vp, vp, vp]
        L.kda_spec_accept.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp]
        L.kda_spec_accept_commit.argtypes = [vp, i64, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                             u32, vp, vp, ctypes.c_int, vp, vp, vp,
                                             ctypes.POINTER(CommitExtras), vp, vp]
        L.kda_conv_compact.argtypes = [ctypes.POINTER(ConvDesc), i32, vp, vp, i32, i32, vp, vp]
        L.kda_selftest_bounded_wait.argtypes = [u32, vp, vp, vp]
        L.kda_slot_copy.argtypes = [ctypes.POINTER(PoolDesc), i32, vp, i32, vp, vp, vp, i32, i32,
                                    vp, sz, vp, vp]
        L.kda_slot_copy_noalloc.argtypes = [ctypes.POINTER(PoolDesc), i32, vp, i32, vp, vp, vp,
                                            i32, i32, vp, vp]
        L.kda_slot_copy_noalloc.restype = ctypes.c_int
        L.kda_chunk_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.kda_chunk_prefill_workspace_size.restype = sz
        L.kda_slot_copy_workspace_size.argtypes = [i64]
        L.kda_slot_copy_workspace_size.restype = sz
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_abi_version.restype = i32
        for f in ("kda_chunk_prefill", "kda_recurrent_decode", "kda_spec_verify",
                  "kda_spec_accept", "kda_spec_commit", "kda_spec_accept_commit",
                  "kda_conv_compact", "kda_slot_copy", "kda_selftest_bounded_wait"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def kda_abi_version() -> int:
    return int(lib().kda_abi_version())


# --------------------------------------------------------------------------
# marshalling helpers


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("libkda takes contiguous CUDA tensors")
    return t.data_ptr()


def _p_any(t):
    """Device pointer of a CUDA tensor whose layout the caller describes itself."""
    if not t.is_cuda:
        raise ValueError("libkda takes CUDA tensors")
    return t.data_ptr()


def _dt(t) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _acts(*ts) -> int:
    """The one activation dtype of the given tensors (bf16 or fp32): the C ABI takes a
    single in_dtype for q, k, v, beta and gate, so a mix is rejected here."""
    dts = {t.dtype for t in ts if t is not None}
    if len(dts) != 1:
        raise ValueError(f"activations must share one dtype, got {sorted(map(str, dts))}")
    return _dt(next(t for t in ts if t is not None))


def _idx(t, name):
    """Device pointer of an int32 index tensor (or None)."""
    if t is not None and isinstance(t, torch.Tensor) and t.dtype != torch.int32:
        raise ValueError(f"{name} must be an int32 tensor, got {t.dtype}")
    return _p(t)


def _f32(t, name):
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be an fp32 tensor, got {t.dtype}")
    return _p(t)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _state_flag(*states) -> int:
    """The state-type flag bit for the given state tensors (None entries are
    ignored); every one of them must have the same dtype."""
    dts = {t.dtype for t in states if t is not None}
    if len(dts) > 1:
        raise ValueError(f"state tensors of different dtypes: {dts}")
    dt = dts.pop() if dts else torch.float32
    if dt == torch.float32:
        return 0
    if dt == torch.bfloat16:
        return KDA_STATE_BF16
    if dt == torch.float16:
        return KDA_STATE_F16
    raise ValueError(f"unsupported state dtype {dt}")


def _check(status: int, where: str):
    if status != 0:
        raise KdaError(status, where)


# --------------------------------------------------------------------------
# entry points


def kda_chunk_prefill_workspace_size(T_tot, N, H, dk=128, dv=128, chunk=64) -> int:
    return int(lib().kda_chunk_prefill_workspace_size(T_tot, N, H, dk, dv, chunk))


def kda_slot_copy_workspace_size(num_slots) -> int:
    """Workspace bytes of kda_slot_copy for pools whose smallest slot count is num_slots."""
    return int(lib().kda_slot_copy_workspace_size(num_slots))


def kda_chunk_prefill(q, k, v, beta_raw, gate_raw, cu_seqlens, out, *, state_pool=None,
                      init_slot=None, final_slot=None, track_chunk_idx=None, track_state=None,
                      scale=1.0, flags=0, chunk=64, workspace=None, dev_status=None, stream=None):
    """Chunked prefill over packed sequences (see include/kda.h)."""
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.shape[0] - 1
    M = 0 if track_chunk_idx is None else int(track_chunk_idx.shape[-1])
    P = 0 if state_pool is None else int(state_pool.shape[0])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    in_dt = _acts(q, k, v, beta_raw, gate_raw)
    st = lib().kda_chunk_prefill(
        _p(q), _p(k), _p(v), _p(beta_raw), _p(gate_raw), in_dt, _idx(cu_seqlens, "cu_seqlens"),
        N, T_tot, H, dk, dv, chunk, float(scale),
        int(flags) | _state_flag(state_pool, track_state), _p(state_pool), P,
        _idx(init_slot, "init_slot"), _idx(final_slot, "final_slot"),
        _idx(track_chunk_idx, "track_chunk_idx"), M, _p(track_state), _p(out), _dt(out),
        _p(workspace), ws_bytes, _idx(dev_status, "dev_status"), _stream(stream))
    _check(st, "kda_chunk_prefill")


def kda_recurrent_decode(q, k, v, beta_raw, gate_raw, state_pool, slot, out, *, scale=1.0,
                         flags=0, dev_status=None, stream=None):
    """One token per request, in place on state_pool[slot] (see include/kda.h)."""
    R, H, dk = q.shape
    dv = v.shape[2]
    in_dt = _acts(q, k, v, beta_raw, gate_raw)
    st = lib().kda_recurrent_decode(
        _p(q), _p(k), _p(v), _p(beta_raw), _p(gate_raw), in_dt, R, H, dk, dv, float(scale),
        int(flags) | _state_flag(state_pool), _p(state_pool), int(state_pool.shape[0]),
        _idx(slot, "slot"), _p(out), _dt(out), _idx(dev_status, "dev_status"), _stream(stream))
    _check(st, "kda_recurrent_decode")


def kda_spec_verify(q, k, v, beta_raw, gate_raw, state_pool, ckpt_slot, rec_u, rec_kg, out, *,
                    K, q_len=None, scale=1.0, flags=0, dev_status=None, stream=None):
    """K speculative positions per request from one checkpoint (see include/kda.h)."""
    RK, H, dk = q.shape
    dv = v.shape[2]
    K = int(K)
    if K < 0 or (K > 0 and RK % K):
        raise ValueError(f"q has {RK} rows, not a multiple of K = {K}")
    R = RK // K if K > 0 else int(ckpt_slot.numel())  # K = 0 launches nothing
    in_dt = _acts(q, k, v, beta_raw, gate_raw)
    if rec_kg.dtype != q.dtype:
        raise ValueError(f"rec_kg holds the activations' dtype {q.dtype}, got {rec_kg.dtype}")
    st = lib().kda_spec_verify(
        _p(q), _p(k), _p(v), _p(beta_raw), _p(gate_raw), in_dt, R, K, _idx(q_len, "q_len"), H,
        dk, dv, float(scale), int(flags) | _state_flag(state_pool), _p(state_pool),
        int(state_pool.shape[0]), _idx(ckpt_slot, "ckpt_slot"), _f32(rec_u, "rec_u"),
        _p(rec_kg), _p(out), _dt(out), _idx(dev_status, "dev_status"), _stream(stream))
    _check(st, "kda_spec_verify")


def kda_spec_accept(tokens, sampled, num_accepted, *, q_len=None, next_token=None,
                    dev_status=None, stream=None):
    """Accepted length per request from draft vs sampled ids (see include/kda.h).

    tokens, sampled: int32 CUDA tensors [R, K]."""
    R, K = tokens.shape
    st = lib().kda_spec_accept(_idx(tokens, "tokens"), _idx(sampled, "sampled"),
                               _idx(q_len, "q_len"), R, K, _idx(num_accepted, "num_accepted"),
                               _idx(next_token, "next_token"), _idx(dev_status, "dev_status"),
                               _stream(stream))
    _check(st, "kda_spec_accept")


def kda_spec_commit(state_pool, ckpt_slot, num_accepted, rec_u, rec_kg, *, K, dst_slot=None,
                    q_len=None, flags=0, plan_out=None, dev_status=None, stream=None):
    """Closed-form rebuild at the accepted length (see include/kda.h)."""
    P, H, dv, dk = state_pool.shape
    R = ckpt_slot.shape[0]
    st = lib().kda_spec_commit(
        _p(state_pool), P, _idx(ckpt_slot, "ckpt_slot"), _idx(dst_slot, "dst_slot"),
        _idx(num_accepted, "num_accepted"), _idx(q_len, "q_len"), R, K, H, dk, dv,
        int(flags) | _state_flag(state_pool), _f32(rec_u, "rec_u"), _p(rec_kg), _dt(rec_kg),
        _idx(plan_out, "plan_out"), _idx(dev_status, "dev_status"), _stream(stream))
    _check(st, "kda_spec_commit")


def _conv_descs(convs):
    n = 0 if convs is None else len(convs)
    descs = (ConvDesc * max(n, 1))()
    for i, t in enumerate(convs or ()):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError("conv tensors need contiguous rows")
        descs[i] = ConvDesc(_p_any(t), t.stride(0) * t.element_size(),
                            t.shape[2] * t.element_size(), t.shape[1], t.shape[0])
    return descs, n


def kda_spec_accept_commit(state_pool, ckpt_slot, tokens, sampled, rec_u, rec_kg, *,
                           dst_slot=None, q_len=None, flags=0, num_accepted=None,
                           next_token=None, plan_out=None, convs=None, conv_slot=None,
                           conv_keep=0, seq_len0=None, block_size=0, block_slot=None,
                           block_idx_out=None, dev_status=None, stream=None):
    """Accepted lengths from token ids, the closed-form rebuild and, optionally, the
    short-convolution windows and the align-mode boundary states, one launch (see
    include/kda.h).  tokens, sampled: int32 CUDA tensors [R, K]; convs: list of CUDA
    tensors [num_slots, rows, channels]."""
    P, H, dv, dk = state_pool.shape
    R, K = tokens.shape
    descs, n = _conv_descs(convs)
    extras = CommitExtras(descs, _idx(conv_slot, "conv_slot"), _idx(seq_len0, "seq_len0"),
                          _idx(block_slot, "block_slot"), _idx(block_idx_out, "block_idx_out"),
                          n, int(conv_keep), int(block_size), 0)
    st = lib().kda_spec_accept_commit(
        _p(state_pool), P, _idx(ckpt_slot, "ckpt_slot"), _idx(dst_slot, "dst_slot"),
        _idx(tokens, "tokens"), _idx(sampled, "sampled"), _idx(q_len, "q_len"), R, K, H, dk, dv,
        int(flags) | _state_flag(state_pool), _f32(rec_u, "rec_u"), _p(rec_kg), _dt(rec_kg),
        _idx(num_accepted, "num_accepted"), _idx(next_token, "next_token"),
        _idx(plan_out, "plan_out"), ctypes.byref(extras), _idx(dev_status, "dev_status"),
        _stream(stream))
    _check(st, "kda_spec_accept_commit")


def kda_conv_compact(convs, slot, num_accepted, keep, *, dev_status=None, stream=None):
    """Short-convolution window after acceptance on every conv tensor (see include/kda.h).

    convs: list of CUDA tensors [num_slots, rows, channels] (slot = first dimension, a row
    contiguous)."""
    descs, n = _conv_descs(convs)
    R = int(slot.numel())
    st = lib().kda_conv_compact(descs, n, _idx(slot, "slot"), _idx(num_accepted, "num_accepted"),
                                R, int(keep), _idx(dev_status, "dev_status"), _stream(stream))
    _check(st, "kda_conv_compact")


def kda_selftest_bounded_wait(polls, dev_status, cycles=None, stream=None):
    """Diagnostic: the kernels' bounded wait on a barrier nothing arrives on (see
    include/kda.h).  dev_status: int32 CUDA tensor; cycles: int64 CUDA tensor or None."""
    st = lib().kda_selftest_bounded_wait(int(polls), _idx(dev_status, "dev_status"), _p(cycles),
                                         _stream(stream))
    _check(st, "kda_selftest_bounded_wait")


def kda_slot_copy(pools, clear_slots, src_slots, dst_offsets, dst_slots, workspace, *,
                  dev_status=None, stream=None):
    """Clear / copy / fan out slots on every pool in one launch (see include/kda.h).

    pools: list of CUDA tensors [num_slots, ...] (slot = first dimension)."""
    descs, n, sets = _slot_sets(pools, clear_slots, src_slots, dst_offsets, dst_slots)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().kda_slot_copy(descs, n, *sets, _p(workspace), ws_bytes,
                             _idx(dev_status, "dev_status"), _stream(stream))
    _check(st, "kda_slot_copy")


def kda_slot_copy_noalloc(pools, clear_slots, src_slots, dst_offsets, dst_slots, *,
                          dev_status=None, stream=None):
    """The slot copy with the library's own fixed check scratch instead of a workspace
    (pools of at most KDA_SLOT_COPY_NOALLOC_MAX_SLOTS slots; see include/kda.h)."""
    descs, n, sets = _slot_sets(pools, clear_slots, src_slots, dst_offsets, dst_slots)
    st = lib().kda_slot_copy_noalloc(descs, n, *sets, _idx(dev_status, "dev_status"),
                                     _stream(stream))
    _check(st, "kda_slot_copy_noalloc")


def _slot_sets(pools, clear_slots, src_slots, dst_offsets, dst_slots):
    """Pool descriptors and the (pointer, count) arguments of the slot sets."""
    n = len(pools)
    descs = (PoolDesc * max(n, 1))()
    for i, t in enumerate(pools):
        descs[i] = PoolDesc(_p(t), t.stride(0) * t.element_size(),
                            t[0].numel() * t.element_size(), t.shape[0])
    n_clear = 0 if clear_slots is None else int(clear_slots.numel())
    n_src = 0 if src_slots is None else int(src_slots.numel())
    n_dst = 0 if dst_slots is None else int(dst_slots.numel())
    sets = (_idx(clear_slots, "clear_slots"), n_clear, _idx(src_slots, "src_slots"),
            _idx(dst_offsets, "dst_offsets"), _idx(dst_slots, "dst_slots"), n_src, n_dst)
    return descs, n, sets
