"""Planted mistakes in copies of the oracle must each fail at least one pin.

Every mutant below is a plausible slip (a dropped term, a wrong sign, a
transposed axis, an off-by-one in time, a forgotten input).  Each is applied
to a private copy of oracle.c, compiled with gcc, swapped in for the real
library, and run through the pin checks of test_oracle.py.  The real oracle is
never modified.
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "decay_on_columns": ("Scol[i] = exp(g[t * dk + i]) * Scol[i]",
                         "Scol[i] = exp(g[t * dk + (j % dk)]) * Scol[i]"),
    "drop_kv_term": ("Scol[i] = exp(g[t * dk + i]) * Scol[i] + k[t * dk + i] * vtj;",
                     "Scol[i] = exp(g[t * dk + i]) * Scol[i] + 0.0 * vtj;"),
    "kv_sign": ("Scol[i] = exp(g[t * dk + i]) * Scol[i] + k[t * dk + i] * vtj;",
                "Scol[i] = exp(g[t * dk + i]) * Scol[i] - k[t * dk + i] * vtj;"),
    "output_uses_key": ("acc += q[t * dk + i] * Scol[i];", "acc += k[t * dk + i] * Scol[i];"),
    "ignore_S0": ("Scol[i] = c->S0 ? c->S0[bh * dk * dv + i * dv + j] : 0.0;",
                  "Scol[i] = 0.0;"),
    "dg_without_alpha": ("a * sdg;", "sdg;"),
    "dg_uses_current_state": ("sdg += A[j] * Sp[j];", "sdg += A[j] * St[j];"),
    "dq_uses_previous_state": ("sdq += dO[t * dv + j] * St[j];",
                               "sdq += dO[t * dv + j] * Sp[j];"),
    "dv_uses_query": ("sdv += k[t * dk + i] * A[i];", "sdv += q[t * dk + i] * A[i];"),
    "dv_ignores_dS_final": ("for (int64_t i = 0; i < dk; ++i) A[i] = c->dSf ? "
                            "c->dSf[bh * dk * dv + i * dv + j] : 0.0;",
                            "for (int64_t i = 0; i < dk; ++i) A[i] = 0.0;"),
    "checkpoint_off_by_one": ("memcpy(blk, ckpt + b * dv, dv * sizeof(double));",
                              "memcpy(blk, ckpt + (b > 0 ? b - 1 : 0) * dv, "
                              "dv * sizeof(double));"),
    "adjoint_decays_late": ("for (int64_t j = 0; j < dv; ++j) A[j] *= a; /* A = diag(alpha_t) A */",
                            "for (int64_t j = 0; j < dv; ++j) A[j] *= (t > t0 ? a : 1.0);"),
    "dk_sign": ("sdk += A[j] * v[t * dv + j];", "sdk -= A[j] * v[t * dv + j];"),
}

PIN_CHECKS = [
    pins.test_hand_scalar_case,
    pins.test_hand_2x2_case,
    pins.test_alpha_one_is_causal_linear_attention,
    pins.test_closed_form_constant_inputs_long_T,
    lambda: pins.test_recurrence_equals_segmented_chunked_form(4, 2, 16),
    pins.test_gradients_match_central_differences,
    pins.test_gradients_across_checkpoint_blocks,
    pins.test_dlog_alpha_identity,
]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mpath = tmp_path / "oracle_mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-pthread", str(mpath),
                           "-o", str(so), "-lm"])
    lib = oracle.configure(ctypes.CDLL(str(so)))
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = []
    for chk in PIN_CHECKS:
        try:
            chk()
        except AssertionError:
            caught.append(getattr(chk, "__name__", "chunked"))
    assert caught, f"no pin caught the planted mistake {name}"
