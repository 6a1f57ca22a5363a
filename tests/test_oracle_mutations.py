"""The oracle's pins must catch plausible mistakes in its arithmetic.

Each case plants one mistake in a copy of the oracle's C source, builds that copy with the
same compiler flags, and runs every pin of test_oracle_pins.py against it: at least one pin
must fail.  The unmodified source, built the same way, must pass them all.  The planted
mistakes stay within the buffers the oracle is given (no case reads out of bounds).
"""
import inspect
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sparse_mla_oracle.c")

# (name, exact text in the oracle source, replacement)
MUTATIONS = [
    ("scale dropped", "logit[s] = sm_scale * dot;", "logit[s] = dot;"),
    ("sink sign", "den += exp((double)attn_sink[h] - m);", "den += exp(-(double)attn_sink[h] - m);"),
    ("sink left out of O", "o[d] = acc / den;", "o[d] = acc / se;"),
    ("sink inside lse", "lse_row[h] = m + log(se);", "lse_row[h] = m + log(den);"),
    ("lse in base 2", "lse_row[h] = m + log(se);", "lse_row[h] = m + log2(se);"),
    ("max_logits unscaled", "max_row[h] = m;", "max_row[h] = m / sm_scale;"),
    ("empty-row lse sign", "lse_row[h] = INFINITY;", "lse_row[h] = -INFINITY;"),
    ("head index ignored", "const uint16_t* qh = q_row + (int64_t)h * d_qk;",
     "const uint16_t* qh = q_row;"),
    ("V from the wrong columns", "acc += w[s] * bf16_to_double(rows_buf[s][d]);",
     "acc += w[s] * bf16_to_double(rows_buf[s][d_qk - d_v + d]);"),
    ("weights not shifted by the max", "w[s] = exp(logit[s] - m);", "w[s] = exp(logit[s]);"),
    ("index 0 treated as invalid",
     "if (idx < 0 || (int64_t)idx >= c->s_kv) return NULL;",
     "if (idx <= 0 || (int64_t)idx >= c->s_kv) return NULL;"),
    ("topk_length ignored", "int64_t L = row_length(topk_length, t, topk);", "int64_t L = topk;"),
    ("paged offset within a page", "int64_t row = page * c->page_block + idx % c->page_block;",
     "int64_t row = page * c->page_block + (idx + 1) % c->page_block;"),
    ("paged block table ignored",
     "int64_t page = c->block_table[b * c->max_blocks + blk];",
     "int64_t page = b * c->max_blocks + blk;"),
    ("tail length off by one", "L = j + 1;", "L = j;"),
    ("paged table bound clamped instead of masked",
     "if (blk >= c->max_blocks) return NULL;", "if (blk >= c->max_blocks) blk = c->max_blocks - 1;"),
    ("unmapped page read as page 0", "if (page < 0) return NULL;", "if (page < 0) page = 0;"),
    ("off-pool row clamped instead of masked",
     "if (row >= c->pool_rows) return NULL;", "if (row >= c->pool_rows) row = c->pool_rows - 1;"),
]


def _pin_calls():
    """Every pin of test_oracle_pins.py with each of its parameter sets."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        params = [p for p in inspect.signature(fn).parameters if p != "orc"]
        marks = getattr(fn, "pytestmark", [])
        grids = [m for m in marks if m.name == "parametrize"]
        combos = [{}]
        for g in grids:
            argnames = [a.strip() for a in g.args[0].split(",")] if isinstance(g.args[0], str) else list(g.args[0])
            new = []
            for c in combos:
                for v in g.args[1]:
                    vv = v if len(argnames) > 1 else (v,)
                    new.append(dict(c, **dict(zip(argnames, vv))))
            combos = new
        for c in combos:
            assert set(c) == set(params), (name, c, params)
            calls.append((name, fn, c))
    return calls


PIN_CALLS = _pin_calls()


def _build_variant(tmp_path, tag, text):
    src = tmp_path / f"{tag}.c"
    src.write_text(text)
    lib = tmp_path / f"lib{tag}.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-shared", "-fPIC", "-o", str(lib), str(src), "-lm"],
                   check=True)
    return oracle.Variant(str(lib))


def _failing_pins(variant):
    failed = []
    for name, fn, kw in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                fn(variant, **kw)
        except Exception:  # an assertion, or a wrong shape / NaN tripping a numpy check
            failed.append(name)
    return failed


def test_unmodified_source_passes_every_pin(tmp_path):
    assert len(PIN_CALLS) > 20
    variant = _build_variant(tmp_path, "clean", open(SRC).read())
    assert _failing_pins(variant) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not found exactly once: {old}"
    variant = _build_variant(tmp_path, "mut", text.replace(old, new))
    failed = _failing_pins(variant)
    assert failed, f"no pin caught the planted mistake '{name}'"
