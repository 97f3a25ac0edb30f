"""Plant plausible mistakes in a copy of the oracle source and check that every
one of them fails at least one pin.  The mistakes are planted on the CPU in a
temporary copy; the real oracle is untouched."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "la_oracle.c")

# (name, exact text in la_oracle.c, replacement)
MUTANTS = [
    ("phi_negative_branch_is_elu", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x + 1.0 : exp(x) - 1.0;"),
    ("phi_dropped_plus_one", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x : exp(x);"),
    ("dphi_missing_exp", "return x > 0.0 ? 1.0 : exp(x);", "return 1.0;"),
    ("causal_mask_strict", "int jend = causal ? i : N - 1;", "int jend = causal ? i - 1 + (i == 0) : N - 1;"),
    ("step_reads_before_update", "double den = 0.0;\n        for (int d = 0; d < Dk; ++d) den += phi(qh[d]) * zh[d];",
     "double den = 0.0;\n        for (int d = 0; d < Dk; ++d) den += phi(qh[d]) * (zh[d] - phi(kh[d]));"),
    ("assoc_transposed_state", "num += qt[d] * S[(size_t)d * Dv + m];", "num += qt[d] * S[(size_t)m * Dk + d];"),
    ("chunk_den_drops_rowsum", "for (int b = 0; b < n; ++b) den += A[(size_t)a * C + b];", ""),
    ("chunk_state_drops_z", "z[d] += kb[d];", "z[d] += 0.0;"),
    ("bwd_g_sign", "g[i] = -od / den;", "g[i] = od / den;"),
    ("bwd_reverse_uses_k", "R[(size_t)d * Dv + m] += qt[d] * P[(size_t)j * Dv + m];",
     "R[(size_t)d * Dv + m] += kt[d] * P[(size_t)j * Dv + m];"),
    ("bwd_direct_dv_no_den", "for (int m = 0; m < Dv; ++m) dvh[(size_t)j * Dv + m] += w * dOi[m] / den[i];\n            }\n        }\n        const double* qh",
     "for (int m = 0; m < Dv; ++m) dvh[(size_t)j * Dv + m] += w * dOi[m];\n            }\n        }\n        const double* qh"),
    ("bwd_dq_drops_gz", "double s = g[i] * z[d];", "double s = 0.0;"),
    ("noncausal_bwd_dk_uses_k", "dkt[(size_t)j * Dk + d] += gw * qt[(size_t)i * Dk + d];\n                }\n                for (int m = 0; m < Dv; ++m) dvh[(size_t)j * Dv + m] += w * dOi[m] / den[i];\n            }\n        }\n        const double* qh = q + IDX3(h, 0, 0, N, Dk);\n        const double* kh = k + IDX3(h, 0, 0, N, Dk);\n        for (size_t t = 0; t < (size_t)N * Dk; ++t) {\n            dq[IDX3(h, 0, 0, N, Dk) + t] = dqt[t] * dphi(qh[t]);\n            dk[IDX3(h, 0, 0, N, Dk) + t] = dkt[t] * dphi(kh[t]);\n        }\n        free(qt); free(kt); free(den); free(oh); free(dqt); free(dkt);\n    }\n}\n",
     "dkt[(size_t)j * Dk + d] += gw * kt[(size_t)j * Dk + d];\n                }\n                for (int m = 0; m < Dv; ++m) dvh[(size_t)j * Dv + m] += w * dOi[m] / den[i];\n            }\n        }\n        const double* qh = q + IDX3(h, 0, 0, N, Dk);\n        const double* kh = k + IDX3(h, 0, 0, N, Dk);\n        for (size_t t = 0; t < (size_t)N * Dk; ++t) {\n            dq[IDX3(h, 0, 0, N, Dk) + t] = dqt[t] * dphi(qh[t]);\n            dk[IDX3(h, 0, 0, N, Dk) + t] = dkt[t] * dphi(kh[t]);\n        }\n        free(qt); free(kt); free(den); free(oh); free(dqt); free(dkt);\n    }\n}\n"),
    ("noncausal_assoc_bwd_g_sign", "g -= P[m] * num[m] / den;", "g += P[m] * num[m] / den;"),
    ("noncausal_assoc_bwd_dk_drops_r", "double rv = r[d];", "double rv = 0.0;"),
    ("noncausal_assoc_bwd_r_from_k", "r[d] += g * qi[d];", "r[d] += g * kt[(size_t)i * Dk + d];"),
    ("retention_decay_exponent_plus_one", "const double w = powi(gamma[h], i - j) * dot(",
     "const double w = powi(gamma[h], i - j + 1) * dot("),
    ("retention_step_decays_after_adding",
     "Sh[(size_t)d * Dv + m] = gamma[h] * Sh[(size_t)d * Dv + m] + kh[d] * vh[m];",
     "Sh[(size_t)d * Dv + m] = gamma[h] * (Sh[(size_t)d * Dv + m] + kh[d] * vh[m]);"),
    ("retention_chunk_carry_exponent", "const double carry = powi(g, a + 1);", "const double carry = powi(g, a);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    if name == "noncausal_bwd_dk_uses_k":
        # the anchor ends the file's last function; replace that (last) occurrence only
        i = src.rfind(old)
        mutated = src[:i] + new + src[i + len(old):]
    else:
        mutated = src.replace(old, new, 1)
    assert mutated != src
    path = tmp_path / "la_oracle_mutant.c"
    path.write_text(mutated)
    so = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(oracle.load_library(so))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
        except pytest.skip.Exception:  # a pin that cannot run here (sympy missing) catches nothing
            pass
    assert failed, "planted mistake %s passed every pin" % name
