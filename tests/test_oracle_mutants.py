"""The pins are strong enough: every plausible slip planted in a COPY of the
oracle source (a dropped term, a wrong sign, index or operand) is caught by
at least one pin.  Mutants are compiled into a temporary directory; the real
oracle is never modified."""
import os
import subprocess

import pytest

import oracle
from tests import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "smqa_oracle.c")

# (name, exact text in the oracle, replacement)
MUTANTS = [
    ("sink dropped from Z", "double Z = exp(sink_h - M);", "double Z = 0.0;"),
    ("natural-log LSE", "(M + log(Z)) / log(2.0)", "(M + log(Z))"),
    ("logit scale dropped", "p[j] = c * acc;", "p[j] = acc;"),
    ("normalisation dropped", "for (int j = 0; j < topk; ++j) p[j] /= Z;", ""),
    ("row 0 treated as masked", "return r >= 0 && r < S_kv;", "return r > 0 && r < S_kv;"),
    ("batch offset of kv dropped", "load_row(kv, ((size_t)b * S_kv + (size_t)r) * D, D, dst);",
     "load_row(kv, ((size_t)r) * D, D, dst);"),
    ("O summed over the query", "orow[d] += p[j] * v[d];", "orow[d] += p[j] * qh[d];"),
    ("g sign flipped", "g[j] = p[j] * (dP - Delta);", "g[j] = p[j] * (dP + Delta);"),
    ("Delta from q not O", "Delta += doh[d] * oh[d];", "Delta += doh[d] * qh[d];"),
    ("scale dropped in dQ", "dqrow[d] += sm_scale * g[j] * k[d];", "dqrow[d] += g[j] * k[d];"),
    ("q and dO swapped in dKV", "sm_scale * g[j] * qh[d] + p[j] * doh[d]",
     "sm_scale * g[j] * doh[d] + p[j] * qh[d]"),
    ("p*dO term dropped from dKV", "sm_scale * g[j] * qh[d] + p[j] * doh[d]",
     "sm_scale * g[j] * qh[d]"),
    ("dKV scattered to the slot number",
     "dkv + ((size_t)b * S_kv + (size_t)idx_row[j]) * D",
     "dkv + ((size_t)b * S_kv + (size_t)j) * D"),
    ("dsink sign flipped", "dsink[h] += -psink * Delta;", "dsink[h] += psink * Delta;"),
    ("absolute floor on dP - Delta", "g[j] = p[j] * (dP - Delta);",
     "g[j] = fabs(dP - Delta) < 1e-7 ? 0.0 : p[j] * (dP - Delta);"),
    ("indexer weight dropped", "dqrow[d] += wh * gj * kj[d];", "dqrow[d] += gj * kj[d];"),
    ("indexer gate inverted", "if (l > 0.0)\n                            for (int d = 0; d < D; ++d) dqrow",
     "if (l < 0.0)\n                            for (int d = 0; d < D; ++d) dqrow"),
    ("indexer ReLU value instead of its slope", "dqrow[d] += wh * gj * kj[d];",
     "dqrow[d] += wh * gj * l * kj[d];"),
    ("indexer key row by slot number",
     "if (valid[j]) load_row(k, (size_t)idx_row[j] * D, D, rows + (size_t)j * D);",
     "if (valid[j]) load_row(k, (size_t)j * D, D, rows + (size_t)j * D);"),
    ("indexer grad_scores of the mirrored slot", "const double gj = g[(size_t)t * topk + j];",
     "const double gj = g[(size_t)t * topk + (topk - 1 - j)];"),
]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant, tmp_path):
    name, old, new = mutant
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mpath), "-o",
                    str(so), "-lm"], check=True)
    lib = oracle.load(str(so))
    caught = []
    for pin in _pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the mutant {name!r}"
