"""Planted mistakes in the oracle: every plausible slip must fail a pin.

Each mutant is one textual change of the oracle's own source (a dropped term,
a flipped sign, an index one off, the wrong operand), compiled (the C
recurrence) or executed (the Python parts) beside the real oracle on the CPU.
The pins of test_oracle_pins.py then run against the mutant, and at least one
of them has to fail.  The real oracle is restored after every mutant.
"""
import inspect
import textwrap

import pytest

import oracle
import test_oracle_pins as pins

# (name, exact text in kda_oracle.c, replacement)
C_MUTANTS = [
    ("decay dropped", "row[i] *= alpha_tmp[i];", "(void)alpha_tmp;"),
    ("correction sign flipped", "double u = beta * (v[c] - xk);", "double u = beta * (v[c] + xk);"),
    ("beta dropped", "double u = beta * (v[c] - xk);", "double u = (v[c] - xk);"),
    ("output read before the write",
     "row[i] += (k[i] * nk) * u;\n            o += row[i] * (scale * (q[i] * nq));",
     "o += row[i] * (scale * (q[i] * nq));\n            row[i] += (k[i] * nk) * u;"),
    ("output uses the key", "o += row[i] * (scale * (q[i] * nq));", "o += row[i] * (scale * (k[i] * nk));"),
    ("scale dropped", "o += row[i] * (scale * (q[i] * nq));", "o += row[i] * (q[i] * nq);"),
    ("L2 norm: key not normalised in the write", "row[i] += (k[i] * nk) * u;", "row[i] += k[i] * u;"),
    ("L2 norm: query not normalised", "o += row[i] * (scale * (q[i] * nq));",
     "o += row[i] * (scale * q[i]);"),
    ("L2 norm: commit uses the raw key record",
     "+ (kg[i] * nk) * u[cc];", "+ kg[i] * u[cc];"),
    ("L2 norm: eps dropped", "return 1.0 / sqrt(ss + ORC_L2NORM_EPS);", "return 1.0 / sqrt(ss);"),
    ("softplus term dropped for positive inputs",
     "if (raw > 0.0) return -(raw + log1p(exp(-raw)));",
     "if (raw > 0.0) return -(log1p(exp(-raw)));"),
    ("sigmoid sign flipped", "return 1.0 / (1.0 + exp(-raw));", "return 1.0 / (1.0 + exp(raw));"),
    ("snapshot one chunk early", "const int j = local / c->chunk;",
     "const int j = local / c->chunk + 1;"),
    ("initial state ignored", "if (c->S0)\n        memcpy", "if (0)\n        memcpy"),
    ("verify records the key as the gate", "memcpy(rkg + dk, c->gate + th * dk",
     "memcpy(rkg + dk, c->k + th * dk"),
    ("commit decays with the key record", "alpha[i] = exp(orc_gate(kg[dk + i], c->flags));",
     "alpha[i] = exp(orc_gate(kg[i], c->flags));"),
    ("commit one step short", "for (int t = 0; t < a; ++t) {\n        const double *u = c->rec_u",
     "for (int t = 0; t + 1 < a; ++t) {\n        const double *u = c->rec_u"),
    ("verify runs past q_len", "if (t < ql) {\n            orc_step", "if (t < K) {\n            orc_step"),
]

# (name, oracle function, exact text in its source, replacement)
PY_MUTANTS = [
    ("accept counts one draft too many", "accept", "a_out[r] = kept + 1", "a_out[r] = kept + 2"),
    ("accept compares the wrong position", "accept", "tokens[r, kept + 1] == sampled[r, kept]",
     "tokens[r, kept] == sampled[r, kept]"),
    ("accept: next token one off", "accept", "nxt[r] = sampled[r, kept]",
     "nxt[r] = sampled[r, max(kept - 1, 0)]"),
    ("conv window one row early", "conv_compact", "pl[sl, a:a + keep]", "pl[sl, a - 1:a - 1 + keep]"),
    ("align: boundary at the span start counted", "align_plan", "if hi > L0[r] // block_size:",
     "if hi >= L0[r] // block_size:"),
    ("align: accepted length one off", "align_plan", "a_b[r] = hi * block_size - L0[r]",
     "a_b[r] = hi * block_size - L0[r] - 1"),
    ("plan accepts lengths past q_len", "commit_plan", "0 <= a <= ql", "0 <= a <= K"),
    ("closed form: checkpoint not decayed", "commit_closed_form", "np.exp(suffix)[:, None] * S0.T",
     "S0.T"),
    ("closed form: suffix includes its own step", "commit_closed_form",
     "acc += (np.exp(suffix) * kk[t])", "acc += (np.exp(suffix + g[t]) * kk[t])"),
    ("closed form: raw key record under the L2 norm", "commit_closed_form",
     "kk = qk_rows(np.asarray(rec_k, np.float64), flags)", "kk = np.asarray(rec_k, np.float64)"),
    ("chunk form: diagonal kept in A", "chunked_prefill", "np.tri(L, k=-1)", "np.tri(L, k=0)"),
    ("chunk form: correction sign flipped", "chunked_prefill", "U = Ut - W @ S", "U = Ut + W @ S"),
]


def _pin_calls():
    """Every pin of test_oracle_pins.py with each of its parameter values."""
    out = []
    for name, fn in sorted(vars(pins).items()):
        if not name.startswith("test_") or not callable(fn):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            out.append((name, fn, {}))
            continue
        argname, values = marks[0].args
        for val in values:
            out.append((f"{name}[{val}]", fn, {argname: val}))
    return out


def _failing_pins():
    failed = []
    for name, fn, kw in _pin_calls():
        try:
            fn(**kw)
        except Exception:  # an assertion, or the mutant breaking the computation outright
            failed.append(name)
    return failed


def test_pins_pass_on_the_real_oracle():
    assert _failing_pins() == []


@pytest.mark.parametrize("name,old,new", C_MUTANTS, ids=[m[0] for m in C_MUTANTS])
def test_c_mutant_fails_a_pin(name, old, new, tmp_path, monkeypatch):
    src = oracle._SRC.read_text()
    assert src.count(old) == 1, f"mutant text for '{name}' must occur once"
    msrc = tmp_path / "kda_oracle.c"
    msrc.write_text(src.replace(old, new))
    monkeypatch.setattr(oracle, "_SRC", msrc)
    monkeypatch.setattr(oracle, "_BUILD", tmp_path)
    monkeypatch.setattr(oracle, "_LIB_PATH", tmp_path / "liboracle_mutant.so")
    monkeypatch.setattr(oracle, "_lib", None)
    oracle._load()  # the mutant compiles and loads: a build error must not count as a kill
    assert _failing_pins(), f"no pin fails with '{name}'"


@pytest.mark.parametrize("name,fn_name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_python_mutant_fails_a_pin(name, fn_name, old, new, monkeypatch):
    src = textwrap.dedent(inspect.getsource(getattr(oracle, fn_name)))
    assert src.count(old) == 1, f"mutant text for '{name}' must occur once"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant: {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, fn_name, ns[fn_name])
    assert _failing_pins(), f"no pin fails with '{name}'"
