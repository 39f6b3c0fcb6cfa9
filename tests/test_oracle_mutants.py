"""Plant plausible mistakes in the oracle (on the CPU) and show the pins catch each.

Each mutant is the oracle's C source with one textual edit, compiled to a
temporary library.  A mutant that passes every pin would mean the pins are too
weak to trust the oracle.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "la_oracle.c")

MUTANTS = {
    # phi without the +1 (plain elu: negative weights possible)
    "phi_drops_plus_one": ("return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x : exp(x) - 1.0;"),
    # sign error in the exponential branch
    "phi_wrong_sign": ("return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x + 1.0 : exp(-x);"),
    # recurrence: state built from phi(q) instead of phi(k)
    "state_uses_q": ("Sr[c] += fk[r] * vt[c];", "Sr[c] += fq[r] * vt[c];"),
    # recurrence: denominator from the current key only (dropped accumulation)
    "den_drops_history": ("            double den = 0.0;\n            for (int r = 0; r < dk; ++r)\n                den += fq[r] * z[r];",
                          "            double den = 0.0;\n            for (int r = 0; r < dk; ++r)\n                den += fq[r] * fk[r];"),
    # clamp replaced by a floor of zero
    "no_eps_clamp": ("return den > eps ? den : eps;", "return den > eps ? den : 0.0 * eps + den;"),
    # chunked: transposed state read (dk != dv exposes it)
    "chunked_transposed_state": ("s += fq[r] * state[(size_t)r * dv + c];",
                                 "s += fq[r] * state[((size_t)c * dk + r) % ((size_t)dk * dv)];"),
    # chunked: diagonal dropped from the intra-chunk mask (exclusive causality)
    "chunked_exclusive_mask": ("for (int b = 0; b <= a; ++b) {", "for (int b = 0; b < a; ++b) {"),
    # non-causal: denominator without the key sums
    "noncausal_den_no_z": ("den += fq[r] * zb[r];\n            den = clamp_den(den, eps);\n            double *oi",
                           "den += fq[r];\n            den = clamp_den(den, eps);\n            double *oi"),
    # decode: normaliser accumulates phi(q)
    "decode_z_uses_q": ("            zb[r] += fk[r];\n        }\n        double den",
                        "            zb[r] += fq[r];\n        }\n        double den"),
    # prefill: v index off by one token
    "prefill_v_shifted": ("Sb[(size_t)r * dv + c] += fk[r] * load(v, type, vb + (int64_t)t * dv + c);",
                          "Sb[(size_t)r * dv + c] += fk[r] * load(v, type, vb + (int64_t)((t + 1) % N) * dv + c);"),
    # bf16 widening with the wrong shift
    "bf16_wrong_shift": ("<< 16;", "<< 15;"),
    # decay: the normaliser not decayed
    "decay_z_undecayed": ("z[r] = g * z[r] + fk[r];", "z[r] = z[r] + fk[r];"),
    # decay: the current token decayed too (exponent off by one)
    "decay_current_token_decayed": ("Sr[c] = g * Sr[c] + fk[r] * vt[c];", "Sr[c] = g * (Sr[c] + fk[r] * vt[c]);"),
    # decay, weighted quadratic form: exponent with the wrong sign
    "decay_quadratic_sign": ("pow(g, (double)(i - j))", "pow(g, (double)(j - i))"),
    # decayed decode: normaliser accumulates phi(q)
    "decode_decay_z_uses_q": ("zb[r] = g * zb[r] + fk[r];", "zb[r] = g * zb[r] + fq[r];"),
    # decayed decode: state not decayed
    "decode_decay_state_undecayed": ("Sb[(size_t)r * dv + c] = g * Sb[(size_t)r * dv + c] + fk[r]",
                                     "Sb[(size_t)r * dv + c] = Sb[(size_t)r * dv + c] + fk[r]"),
    # feature maps and the normaliser
    "relu_keeps_negative_part": ("return (x > 0.0 ? x : 0.0) + c;", "return (x > 0.0 ? 0.0 : x) + c;"),
    "identity_drops_shift": ("        return x + c;\n    return la_oracle_phi(x);", "        return x;\n    return la_oracle_phi(x);"),
    "general_always_normalizes": ("            if (normalize) {\n                double den = 0.0;", "            if (1) {\n                double den = 0.0;"),
    "general_ignores_decay": ("        const double g = gamma ? gamma[bh] : 1.0;\n        double *S = calloc", "        const double g = 1.0;\n        double *S = calloc"),
    "prefill_general_undecayed": ("Sb[(size_t)r * dv + c] = g * Sb[(size_t)r * dv + c] +\n", "Sb[(size_t)r * dv + c] = Sb[(size_t)r * dv + c] +\n"),
    "noncausal_general_default_map": ("la_oracle_prefill_state_general(k, v, type, NULL, map, shift, S, z, BH, N, dk, dv);", "la_oracle_prefill_state_general(k, v, type, NULL, 0, shift, S, z, BH, N, dk, dv);"),
    "decode_general_key_from_query": ("fk[r] = phi_map(load(k, type, (int64_t)bh * dk + r), map, shift);", "fk[r] = phi_map(load(q, type, (int64_t)bh * dk + r), map, shift);"),
    # backward pass
    "backward_drops_denominator_term": ("dd[t] = clamped ? 0.0 : -g / d;", "dd[t] = 0.0;"),
    "backward_reverse_state_from_k": ("Rr[c] += fq[r] * dn[(size_t)t * dvd + c];", "Rr[c] += fk[r] * dn[(size_t)t * dvd + c];"),
    "backward_phi_prime_constant": ("    return x > 0.0 ? 1.0 : exp(x);", "    return 1.0;"),
    "backward_dv_from_q": ("s += R[(size_t)r * dvd + c] * fk[r];", "s += R[(size_t)r * dvd + c] * fq[r];"),
    "backward_dq_sign": ("double s = dd[t] * z[r];", "double s = -dd[t] * z[r];"),
    # gated state (one gate per key feature)
    "gated_z_ungated": ("z[r] = at[r] * z[r] + fk[r];", "z[r] = z[r] + fk[r];"),
    "gated_gate_after_update": ("Sr[c] = at[r] * Sr[c] + fk[r] * vt[c];", "Sr[c] = at[r] * (Sr[c] + fk[r] * vt[c]);"),
    "gated_gate_of_previous_token": ("const double *at = alpha + qb + (int64_t)t * dk;",
                                     "const double *at = alpha + qb + (int64_t)(t > 0 ? t - 1 : 0) * dk;"),
    "gated_gate_on_value_axis": ("Sr[c] = at[r] * Sr[c] + fk[r] * vt[c];", "Sr[c] = at[c % dk] * Sr[c] + fk[r] * vt[c];"),
    "gated_quadratic_gate_index_off": ("prod[r] *= alpha[qb + (int64_t)(j + 1) * dk + r];",
                                       "prod[r] *= alpha[qb + (int64_t)j * dk + r];"),
    "gated_decode_z_uses_q": ("zb[r] = ab[r] * zb[r] + fk[r];", "zb[r] = ab[r] * zb[r] + fq[r];"),
    "gated_prefill_ungated": ("Sb[(size_t)r * dv + c] = at[r] * Sb[(size_t)r * dv + c] + fk[r]",
                              "Sb[(size_t)r * dv + c] = Sb[(size_t)r * dv + c] + fk[r]"),
    # FAVOR+ features
    "favor_drops_norm_term": ("out[i * m + r] = exp(dot - 0.5 * nrm) / sqrt((double)m);", "out[i * m + r] = exp(dot) / sqrt((double)m);"),
    "favor_norm_sign": ("out[i * m + r] = exp(dot - 0.5 * nrm) / sqrt((double)m);", "out[i * m + r] = exp(dot + 0.5 * nrm) / sqrt((double)m);"),
    "favor_no_sqrt_m": ("out[i * m + r] = exp(dot - 0.5 * nrm) / sqrt((double)m);", "out[i * m + r] = exp(dot - 0.5 * nrm) / (double)m;"),
    # W [m, d] read as if stored [d, m] (a transposed operand)
    "favor_transposed_projection": ("dot += W[(size_t)r * d + c] * load(x, type, i * d + c);",
                                    "dot += W[(size_t)c * m + r] * load(x, type, i * d + c);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site vanished: " + name
    mutated = src.replace(old, new, 1)
    mpath = tmp_path / "la_oracle.c"
    mpath.write_text(mutated)
    lib_path = str(tmp_path / "libmutant.so")
    import subprocess
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-w", str(mpath),
                    "-o", lib_path, "-lm"], check=True)
    orc = oracle.Oracle(oracle.load(lib_path))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "no pin caught mutant " + name
