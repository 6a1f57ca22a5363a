"""The backward oracle's pins must catch plausible mistakes in its arithmetic.

Each case plants one mistake in a copy of oracle/sparse_mla_bwd_oracle.c, builds it with the
same flags and runs every pin of test_bwd_oracle_pins.py against it: at least one must fail.
The unmodified source, built the same way, must pass them all.  No planted mistake reads or
writes outside the buffers the oracle is given.
"""
import inspect
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_bwd_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sparse_mla_bwd_oracle.c")

MUTATIONS = [
    ("scale dropped from dq", "dqh[d] += sm_scale * ds * ks[d];", "dqh[d] += ds * ks[d];"),
    ("scale dropped from dk", "cs[d] += sm_scale * ds * qh[d];", "cs[d] += ds * qh[d];"),
    ("delta sign", "double ds = pr[s] * (dp[s] - delta);", "double ds = pr[s] * (dp[s] + delta);"),
    ("delta left out", "double ds = pr[s] * (dp[s] - delta);", "double ds = pr[s] * dp[s];"),
    ("dv without p", "for (int d = 0; d < d_v; ++d) cs[d] += pr[s] * doh[d];",
     "for (int d = 0; d < d_v; ++d) cs[d] += doh[d];"),
    ("sink left out of the normaliser", "  z += e_sink;\n", "\n"),
    ("sink gradient sign", "dsink_row[h] = -(e_sink / z) * delta;", "dsink_row[h] = (e_sink / z) * delta;"),
    ("logit scale dropped", "lg[s] = sm_scale * acc;", "lg[s] = acc;"),
    ("dq from q instead of k", "dqh[d] += sm_scale * ds * ks[d];", "dqh[d] += sm_scale * ds * qh[d];"),
    ("index 0 treated as invalid", "if (v >= 0 && (int64_t)v < s_kv) slot_rows[n++] = v;",
     "if (v > 0 && (int64_t)v < s_kv) slot_rows[n++] = v;"),
    ("topk_length ignored", "if (!topk_length) return topk;", "return topk;"),
    ("value columns shifted", "for (int d = 0; d < d_v; ++d) acc += doh[d] * vs[d];",
     "for (int d = 0; d < d_v; ++d) acc += doh[d] * vs[d_qk - d_v + d];"),
]


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn, {}))
            continue
        argnames = [a.strip() for a in marks[0].args[0].split(",")]
        for v in marks[0].args[1]:
            calls.append((name, fn, dict(zip(argnames, v if len(argnames) > 1 else (v,)))))
    return calls


PIN_CALLS = _pin_calls()


def _build_variant(tmp_path, tag, text):
    src = tmp_path / f"{tag}.c"
    src.write_text(text)
    lib = tmp_path / f"lib{tag}.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", str(lib), str(src), "-lm"],
                   check=True)
    return oracle.BwdVariant(str(lib))


def _failing_pins(variant, monkeypatch):
    failed = []
    with monkeypatch.context() as m:
        m.setattr(oracle, "sparse_mla_bwd_f64", variant.sparse_mla_bwd_f64)
        m.setattr(oracle, "sparse_mla_bwd", variant.sparse_mla_bwd)
        for name, fn, kw in PIN_CALLS:
            try:
                with np.errstate(all="ignore"):
                    fn(**kw)
            except Exception:  # an assertion, or a NaN tripping a numpy check
                failed.append(name)
    return failed


def test_unmodified_source_passes_every_pin(tmp_path, monkeypatch):
    assert len(PIN_CALLS) >= 10
    variant = _build_variant(tmp_path, "clean", open(SRC).read())
    assert _failing_pins(variant, monkeypatch) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not found exactly once: {old}"
    variant = _build_variant(tmp_path, "mut", text.replace(old, new))
    assert _failing_pins(variant, monkeypatch), f"no pin caught the planted mistake '{name}'"
