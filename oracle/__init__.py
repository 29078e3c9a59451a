"""fp64 CPU oracle for the KDA recurrent-state path.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only callers.  The product path never imports this
package, and this package imports nothing from the product.

Contents
  * ``prefill``, ``decode``, ``verify``, ``commit`` -- thin ctypes wrappers
    around ``kda_oracle.c``, the token-by-token recurrence in double precision
    (the per-head KDA state update as stated for Kimi Delta Attention:
    S_t = Diag(alpha_t) S_{t-1} + k_t u_t^T, u_t = beta_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t),
    o_t = S_t^T q_t, alpha_t = exp(g_t), g_t = -softplus(raw gate), beta = sigmoid(raw beta)).
  * ``chunked_prefill`` -- a second, independent fp64 evaluation of the same
    recurrence in chunk (WY / UT-transform) form, used only to check that the
    chunk algebra and the recurrence agree.
  * ``commit_closed_form`` -- the closed-form rebuild at accepted length a
    (RecoverSSM page, implementation breakdown step 4: rebuild the state in
    one shot in reverse order, not by re-running the recursion).
  * ``slot_copy`` and ``commit_plan`` -- memcpy and integer semantics.
  * ``accept`` -- the accepted length of each speculative request from its
    draft and sampled token ids (integer semantics).
  * ``conv_compact`` -- the short-convolution window kept after acceptance
    (copy semantics).
  * ``align_plan`` -- the block boundary an accepted span crosses (integer
    semantics); the state there is ``commit`` at that accepted length.

All arrays are float64 numpy arrays (bf16 inputs widened exactly by the
caller).  Layouts follow the library: activations [tokens, heads, channels],
states transposed [.., heads, d_v, d_k].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

GATE_LOG = 1  # gate input holds g itself
BETA_ACT = 2  # beta input holds beta itself
QK_L2NORM = 32  # q and k rows divided by sqrt(sum x^2 + L2NORM_EPS) before use
L2NORM_EPS = 1e-6

BAD_SLOT = 1
BAD_TRACK = 2
BAD_ACCEPT = 4
BAD_SEQLEN = 8

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "kda_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"
_lib = None
_lock = threading.Lock()


def build_library(force: bool = False) -> Path:
    """Compile the C oracle with gcc (ISO C, no FP contraction, no fast-math)."""
    _BUILD.mkdir(exist_ok=True)
    if force or not _LIB_PATH.exists() or _LIB_PATH.stat().st_mtime < _SRC.stat().st_mtime:
        tmp = _BUILD / f"liboracle.{os.getpid()}.so"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", str(_SRC), "-o", str(tmp), "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build_library()))
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            i, u, d, l = ctypes.c_int, ctypes.c_uint, ctypes.c_double, ctypes.c_long
            lib.kda_oracle_prefill.argtypes = [dp, dp, dp, dp, dp, ip, i, i, i, i, d, u, dp, i,
                                               ip, i, dp, dp, dp, i]
            lib.kda_oracle_decode.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, d, u, dp, l, ip,
                                              dp, i]
            lib.kda_oracle_verify.argtypes = [dp, dp, dp, dp, dp, i, i, ip, i, i, i, d, u, dp, l,
                                              ip, dp, dp, dp, i]
            lib.kda_oracle_commit.argtypes = [dp, l, ip, ip, ip, ip, i, i, i, i, i, u, dp, dp, ip,
                                              i]
            for f in (lib.kda_oracle_prefill, lib.kda_oracle_decode, lib.kda_oracle_verify,
                      lib.kda_oracle_commit):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _dp(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


# --------------------------------------------------------------------------
# token-by-token recurrence (C)


def prefill(q, k, v, beta, gate, cu_seqlens, *, scale=1.0, flags=0, S0=None, chunk=64,
            track=None, n_threads=None):
    """Recurrence over packed sequences.

    q, k, gate: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; cu_seqlens: [N+1].
    S0: [N, H, dv, dk] initial states (None = zero).  track: [N, M] chunk
    indices j; snapshot m of sequence n is the state after exactly j*chunk of
    its tokens (-1 = unused).  Returns (out [T,H,dv], S_final [N,H,dv,dk],
    snapshots [N,M,H,dv,dk] (NaN where not written), status bits).
    """
    q, k, v, beta, gate = map(_f64, (q, k, v, beta, gate))
    cu = _i32(cu_seqlens)
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    if track is None:
        track = np.full((N, 0), -1, np.int32)
    track = _i32(track).reshape(N, -1)
    M = track.shape[1]
    S0c = None if S0 is None else _f64(S0).reshape(N, H, dv, dk)
    out = np.zeros((T, H, dv))
    S_final = np.zeros((N, H, dv, dk))
    snap = np.full((N, max(M, 1), H, dv, dk), np.nan)
    st = _load().kda_oracle_prefill(_dp(q), _dp(k), _dp(v), _dp(beta), _dp(gate), _ip(cu), N,
                                    H, dk, dv, float(scale), int(flags), _dp(S0c), int(chunk),
                                    _ip(track), M, _dp(snap), _dp(S_final), _dp(out),
                                    _threads(n_threads))
    return out, S_final, snap[:, :M], st


def decode(q, k, v, beta, gate, pool, slot, *, scale=1.0, flags=0, n_threads=None):
    """One step per request on pool[slot[r]] (updated in place on a copy).

    Returns (out [R,H,dv], new_pool, status)."""
    q, k, v, beta, gate = map(_f64, (q, k, v, beta, gate))
    pool = _f64(pool).copy()
    slot = _i32(slot)
    R, H, dk = q.shape
    dv = v.shape[2]
    out = np.zeros((R, H, dv))
    st = _load().kda_oracle_decode(_dp(q), _dp(k), _dp(v), _dp(beta), _dp(gate), R, H, dk, dv,
                                   float(scale), int(flags), _dp(pool), pool.shape[0], _ip(slot),
                                   _dp(out), _threads(n_threads))
    return out, pool, st


def verify(q, k, v, beta, gate, pool, ckpt, K, *, q_len=None, scale=1.0, flags=0,
           n_threads=None):
    """K speculative steps from pool[ckpt[r]] without writing the pool.

    Inputs are [R*K, H, ..].  Returns (out [R*K,H,dv], rec_u [R,H,K,dv],
    rec_kg [R,H,K,2dk] (= key and raw gate as given), status)."""
    q, k, v, beta, gate = map(_f64, (q, k, v, beta, gate))
    pool = _f64(pool)
    ckpt = _i32(ckpt)
    RK, H, dk = q.shape
    R = RK // K
    dv = v.shape[2]
    ql = None if q_len is None else _i32(q_len)
    out = np.zeros((RK, H, dv))
    rec_u = np.zeros((R, H, K, dv))
    rec_kg = np.zeros((R, H, K, 2 * dk))
    st = _load().kda_oracle_verify(_dp(q), _dp(k), _dp(v), _dp(beta), _dp(gate), R, K, _ip(ql),
                                   H, dk, dv, float(scale), int(flags), _dp(pool), pool.shape[0],
                                   _ip(ckpt), _dp(rec_u), _dp(rec_kg), _dp(out),
                                   _threads(n_threads))
    return out, rec_u, rec_kg, st


def commit(pool, ckpt, num_accepted, rec_u, rec_kg, K, *, dst=None, q_len=None, flags=0,
           n_threads=None):
    """Brute-force re-recursion of the first a recorded steps.

    Returns (new_pool, plan [R,3] = (a or -1, src, dst), status)."""
    pool = _f64(pool).copy()
    ckpt = _i32(ckpt)
    acc = _i32(num_accepted)
    R = ckpt.shape[0]
    _, H, dv, dk = pool.shape
    rec_u = _f64(rec_u).reshape(R, H, K, dv)
    rec_kg = _f64(rec_kg).reshape(R, H, K, 2 * dk)
    dsta = None if dst is None else _i32(dst)
    ql = None if q_len is None else _i32(q_len)
    plan = np.zeros((R, 3), np.int32)
    st = _load().kda_oracle_commit(_dp(pool), pool.shape[0], _ip(ckpt), _ip(dsta), _ip(acc),
                                   _ip(ql), R, K, H, dk, dv, int(flags), _dp(rec_u), _dp(rec_kg),
                                   _ip(plan), _threads(n_threads))
    return pool, plan, st


# --------------------------------------------------------------------------
# activations in numpy (used by the chunk form and the closed form below)


def gate_log(raw, flags=0):
    """g = -softplus(raw) in fp64 (or raw itself under GATE_LOG)."""
    raw = np.asarray(raw, np.float64)
    if flags & GATE_LOG:
        return raw.copy()
    with np.errstate(over="ignore"):
        return np.where(raw > 0, -(raw + np.log1p(np.exp(-np.abs(raw)))),
                        -np.log1p(np.exp(np.minimum(raw, 0.0))))


def beta_act(raw, flags=0):
    raw = np.asarray(raw, np.float64)
    if flags & BETA_ACT:
        return raw.copy()
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-raw))


def qk_rows(x, flags=0):
    """q or k rows as the recurrence uses them: under QK_L2NORM each row (last axis) is
    divided by sqrt(sum x^2 + L2NORM_EPS) (the per-head L2 normalisation of the serving
    configurations, done inside the path); otherwise unchanged."""
    x = np.asarray(x, np.float64)
    if not flags & QK_L2NORM:
        return x
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2NORM_EPS)


# --------------------------------------------------------------------------
# chunk (WY / UT-transform) form, fp64, for agreement checks only


def chunked_prefill(q, k, v, beta, gate, cu_seqlens, *, chunk, scale=1.0, flags=0, S0=None):
    """Same quantity as ``prefill`` evaluated chunk by chunk.

    Within a chunk with inclusive cumulative gate G_t (per key channel):
      A_ts = sum_i k_ti k_si exp(G_ti - G_si), s < t      (strictly lower)
      P_ts = sum_i q_ti k_si exp(G_ti - G_si), s <= t
      T    = (I + Diag(beta) A)^-1
      W    = T Diag(beta) (k * exp(G)),   U~ = T Diag(beta) V
      U    = U~ - W S                     (S = d_k x d_v state entering the chunk)
      O    = (q * exp(G)) S + P U
      S   <- Diag(exp(G_last)) S + (k * exp(G_last - G))^T U
    Returns (out [T,H,dv], S_final [N,H,dv,dk]) -- states in the transposed layout.
    """
    q, k, v, beta, gate = map(_f64, (q, k, v, beta, gate))
    q, k = qk_rows(q, flags), qk_rows(k, flags)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.asarray(cu_seqlens, np.int64)
    N = cu.shape[0] - 1
    g_all = gate_log(gate, flags)
    b_all = beta_act(beta, flags)
    out = np.zeros((T, H, dv))
    S_fin = np.zeros((N, H, dv, dk))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h]).T.copy()
            for c0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                c1 = min(c0 + chunk, int(cu[n + 1]))
                qc, kc, vc = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
                bc = b_all[c0:c1, h]
                G = np.cumsum(g_all[c0:c1, h], axis=0)
                L = c1 - c0
                D = np.exp(G[:, None, :] - G[None, :, :])  # [t, s, i]
                A = np.einsum("ti,si,tsi->ts", kc, kc, D) * np.tri(L, k=-1)
                P = np.einsum("ti,si,tsi->ts", qc * scale, kc, D) * np.tri(L, k=0)
                Tm = np.linalg.inv(np.eye(L) + bc[:, None] * A)
                W = Tm @ (bc[:, None] * (kc * np.exp(G)))
                Ut = Tm @ (bc[:, None] * vc)
                U = Ut - W @ S
                out[c0:c1, h] = (qc * scale * np.exp(G)) @ S + P @ U
                S = np.exp(G[-1])[:, None] * S + (kc * np.exp(G[-1][None, :] - G)).T @ U
            S_fin[n, h] = S.T
    return out, S_fin


# --------------------------------------------------------------------------
# closed-form commit (self-check against the brute-force recursion)


def commit_closed_form(S0, rec_k, rec_gate, rec_u, a, flags=0):
    """S_a = Diag(exp sum_{t<=a} g_t) S_0 + sum_{t<=a} Diag(exp sum_{t<s<=a} g_s) k_t u_t^T.

    S0: [dv, dk] (transposed state); rec_k, rec_gate: [K, dk]; rec_u: [K, dv].
    Built in reverse order with a running suffix sum of the gates, as the
    RecoverSSM commit is described (one-shot rebuild, no re-recursion).
    Returns the transposed state [dv, dk].
    """
    S0 = _f64(S0)
    dv, dk = S0.shape
    g = gate_log(np.asarray(rec_gate, np.float64)[:a], flags)
    kk = qk_rows(np.asarray(rec_k, np.float64), flags)  # records hold k as given
    acc = np.zeros((dk, dv))
    suffix = np.zeros(dk)  # sum_{t<s<=a} g_s
    for t in range(a - 1, -1, -1):
        acc += (np.exp(suffix) * kk[t])[:, None] * np.asarray(rec_u, np.float64)[t][None, :]
        suffix = suffix + g[t]
    return (np.exp(suffix)[:, None] * S0.T + acc).T


# --------------------------------------------------------------------------
# slot copy and commit plan


def slot_copy(pools, clear_slots, src_slots, dst_offsets, dst_slots):
    """memcpy semantics on each pool (array of [num_slots, ...] of any dtype).

    Clears zero the listed slots; source i is copied to dst_slots[dst_offsets[i]
    : dst_offsets[i+1]].  Sources are read before any write, which is what the
    disjointness precondition (destinations distinct and apart from sources and
    clears) makes equivalent to any order.  Returns new copies."""
    outs = []
    for p in pools:
        p0 = np.array(p, copy=True)
        p1 = np.array(p, copy=True)
        for s in clear_slots:
            p1[int(s)] = 0
        for i, s in enumerate(src_slots):
            for d in dst_slots[int(dst_offsets[i]):int(dst_offsets[i + 1])]:
                p1[int(d)] = p0[int(s)]
        outs.append(p1)
    return outs


def commit_plan(ckpt, num_accepted, P, K, dst=None, q_len=None):
    """Plan rows (a, src, dst); a = -1 marks a request the commit skips."""
    R = len(ckpt)
    plan = np.zeros((R, 3), np.int32)
    for r in range(R):
        src = int(ckpt[r])
        d = int(dst[r]) if dst is not None else src
        ql = int(q_len[r]) if q_len is not None else K
        a = int(num_accepted[r])
        ok = 0 <= src < P and 0 <= d < P and 0 <= ql <= K and 0 <= a <= ql
        plan[r] = (a if ok else -1, src, d)
    return plan


def accept(tokens, sampled, K, q_len=None):
    """Runtime accepted length per request (RecoverSSM page, implementation
    breakdown step 4: the commit plan derives the accepted lengths on the GPU,
    and num_accepted_tokens is written straight back to device buffers).

    tokens[r, 0] is the request's last committed token and tokens[r, 1:q_len]
    its drafts; sampled[r, i] is the target model's token for the position
    after i.  Drafts are kept from the front while draft i+1 equals sampled
    token i; the first mismatch ends the run.  The accepted length a counts the
    positions whose update the state keeps: the committed token plus every
    kept draft, so 1 <= a <= q_len.  The next input token is sampled[r, a-1].
    q_len = 0 (a padding row) gives a = 0 and next = -1; q_len outside [0, K]
    gives a = -1, next = -1 and the BAD_ACCEPT status bit.

    Returns (a [R] int32, next [R] int32, status)."""
    tokens = np.asarray(tokens, np.int64)
    sampled = np.asarray(sampled, np.int64)
    R = tokens.shape[0]
    a_out = np.zeros(R, np.int32)
    nxt = np.zeros(R, np.int32)
    status = 0
    for r in range(R):
        ql = int(q_len[r]) if q_len is not None else K
        if ql < 0 or ql > K:
            a_out[r], nxt[r] = -1, -1
            status |= BAD_ACCEPT
            continue
        if ql == 0:
            a_out[r], nxt[r] = 0, -1
            continue
        kept = 0
        while kept < ql - 1 and tokens[r, kept + 1] == sampled[r, kept]:
            kept += 1
        a_out[r] = kept + 1
        nxt[r] = sampled[r, kept]
    return a_out, nxt, status


def conv_compact(pools, slots, num_accepted, keep):
    """Short-convolution history after a speculative step (RecoverSSM page,
    implementation breakdown step 4: the commit compacts the conv history; the
    "state semantics" page: the conv state is a sliding window moved by an
    offset copy).

    Each pool is [num_slots, rows, channels]: a slot's rows 0..keep-1 hold the
    last `keep` inputs before the step, rows keep.. the step's inputs.  After
    a accepted positions the window is the last `keep` inputs of the accepted
    stream, i.e. rows a .. a+keep-1 move to rows 0 .. keep-1 (rows past keep
    are left as they were).  slot < 0 skips the request; slot >= num_slots
    sets BAD_SLOT; a < 0 or a + keep > rows sets BAD_ACCEPT; both skip.
    Sources are read before any write (the ranges overlap when a < keep).
    Returns (new pools, status)."""
    outs = [np.array(pl, copy=True) for pl in pools]
    status = 0
    for i, pl in enumerate(pools):
        n_slots, rows = pl.shape[0], pl.shape[1]
        for r, sl in enumerate(slots):
            sl, a = int(sl), int(num_accepted[r])
            if sl < 0:
                continue
            if sl >= n_slots:
                status |= BAD_SLOT
                continue
            if a < 0 or a + keep > rows:
                status |= BAD_ACCEPT
                continue
            outs[i][sl, :keep] = pl[sl, a:a + keep]
    return outs, status


def align_plan(seq_len0, num_accepted, block_size):
    """Block boundary inside each request's accepted span (RecoverSSM page,
    implementation breakdown step 4: in align mode the commit plan computes
    the runtime accepted lengths and the align boundaries, and the running
    block index is updated).

    A request had seq_len0 tokens before the step and keeps a more; its
    accepted span is positions seq_len0+1 .. seq_len0+a.  Block boundaries are
    the multiples of block_size.  Returns (a_b, block_idx): a_b is the
    accepted length that ends on the last boundary inside the span (the
    state there is the commit at a_b), -1 when the span holds none; block_idx
    is the number of whole blocks after the step, floor((seq_len0 + a) /
    block_size).  A request with seq_len0 < 0 or a < 0 gets (-1, -1)."""
    L0 = np.asarray(seq_len0, np.int64)
    a = np.asarray(num_accepted, np.int64)
    a_b = np.full(L0.shape, -1, np.int32)
    idx = np.full(L0.shape, -1, np.int32)
    for r in range(L0.shape[0]):
        if L0[r] < 0 or a[r] < 0:
            continue
        hi = (L0[r] + a[r]) // block_size
        idx[r] = hi
        if hi > L0[r] // block_size:
            a_b[r] = hi * block_size - L0[r]
    return a_b, idx
