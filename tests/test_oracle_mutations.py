"""Plant plausible slips in a copy of the oracle's C source and check that the
pins catch every one (the pins would otherwise prove nothing).  CPU only: the
mutated copies are built with gcc into a temporary directory."""
import os

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, original text, replacement, which occurrence (0-based))
MUTATIONS = [
    ("phi_dropped_plus_one", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x : exp(x);", 0),
    ("dphi_zero_for_negative", "return x > 0.0 ? 1.0 : exp(x);", "return x > 0.0 ? 1.0 : 0.0;", 0),
    ("quadratic_mask_strict", "for (int j = 0; j <= i; ++j) {\n        double a", "for (int j = 0; j < i; ++j) {\n        double a", 0),
    ("recurrent_off_by_one_key", "        double fk = phi(K[(size_t)i * D + d]);\n        for (int m = 0; m < M; ++m)\n          S[(size_t)d * M + m] = gamma * S[(size_t)d * M + m] + fk * V[(size_t)i * M + m];",
     "        double fk = phi(K[(size_t)(i > 0 ? i - 1 : 0) * D + d]);\n        for (int m = 0; m < M; ++m)\n          S[(size_t)d * M + m] = gamma * S[(size_t)d * M + m] + fk * V[(size_t)(i > 0 ? i - 1 : 0) * M + m];", 0),
    ("bwd_dropped_denominator_term", "double acc = gam[i] * Z[d];", "double acc = 0.0;", 0),
    ("bwd_gamma_sign", "gam[i] = -gv / s;", "gam[i] = gv / s;", 0),
    ("bwd_dropped_r", "        double acc = r[d];\n        for (int m = 0; m < M; ++m) acc += R[(size_t)d * M + m] * V[(size_t)i * M + m];",
     "        double acc = 0.0;\n        for (int m = 0; m < M; ++m) acc += R[(size_t)d * M + m] * V[(size_t)i * M + m];", 0),
    ("bwd_dv_uses_phiq", "acc += R[(size_t)d * M + m] * phi(K[(size_t)i * D + d]);", "acc += R[(size_t)d * M + m] * phi(Q[(size_t)i * D + d]);", 0),
    ("bwd_reverse_sweep_forward", "for (int i = N - 1; i >= 0; --i) {", "for (int i = 0; i < N; ++i) {", 0),
    ("noncausal_ignores_length", "    for (int j = 0; j < L; ++j)\n      for (int d = 0; d < D; ++d) {\n        double fk", "    for (int j = 0; j < N; ++j)\n      for (int d = 0; d < D; ++d) {\n        double fk", 0),
    ("noncausal_bwd_missing_gamma", "double gam = -gv / s;", "double gam = 0.0 * gv / s;", 0),
    ("decode_no_denominator", "yt[m] = acc / den;", "yt[m] = acc;", 0),
    ("decode_transposed_update", "s[(size_t)d * M + m] = gamma * s[(size_t)d * M + m] + fk * vt[m];",
     "s[(size_t)d * M + m] = gamma * s[(size_t)d * M + m] + fk * vt[d % M];", 0),
    # the RetNet decay
    ("decay_z_not_decayed", "Z[d] = gamma * Z[d] + fk;", "Z[d] = Z[d] + fk;", 0),
    ("decay_exponent_flipped", "a *= pow(gamma, (double)(i - j));", "a *= pow(gamma, (double)(j - i));", 0),
    ("decay_reverse_sum_undecayed", "R[(size_t)d * M + m] = gamma * R[(size_t)d * M + m] + fqd * gt[(size_t)i * M + m];",
     "R[(size_t)d * M + m] = R[(size_t)d * M + m] + fqd * gt[(size_t)i * M + m];", 0),
    ("decay_r_undecayed", "r[d] = gamma * r[d] + gam[i] * fqd;", "r[d] = r[d] + gam[i] * fqd;", 0),
    ("decay_quadratic_grad_undecayed", "da *= pow(gamma, (double)(i - j));", "da *= 1.0;", 0),
    ("decay_decode_z_not_decayed", "z[d] = gamma * z[d] + fk;", "z[d] = z[d] + fk;", 0),
    ("decay_squared", "S[(size_t)d * M + m] = gamma * S[(size_t)d * M + m] + fk * V[(size_t)i * M + m];",
     "S[(size_t)d * M + m] = gamma * gamma * S[(size_t)d * M + m] + fk * V[(size_t)i * M + m];", 0),
    # the degree-2 polynomial kernel
    ("poly_sim_not_squared", "        row[j] = dot * dot;", "        row[j] = dot;", 0),
    ("poly_grad_factor_dropped", "const double w = 2.0 * da * dots[j];", "const double w = da * dots[j];", 0),
    ("poly_dk_uses_k", "dK[(size_t)j * D + d] += w * Q[(size_t)i * D + d];", "dK[(size_t)j * D + d] += w * K[(size_t)j * D + d];", 0),
    ("poly_dv_unsquared", "dV[(size_t)j * M + m] += dots[j] * dots[j] * gt[m];", "dV[(size_t)j * M + m] += dots[j] * gt[m];", 0),
    ("prefill_starts_from_zero", "memcpy(sl, st, sizeof(double) * (size_t)D * M);", "memset(sl, 0, sizeof(double) * (size_t)D * M);", 0),
    ("prefill_den_without_z0", "for (int d = 0; d < D; ++d) zl[d] = zt[d];", "for (int d = 0; d < D; ++d) zl[d] = 0.0 * zt[d];", 0),
    ("prefill_state_not_returned", "for (size_t e = 0; e < (size_t)D * M; ++e) st[e] = sl[e];", "for (size_t e = 0; e < (size_t)D * M; ++e) (void)sl[e];", 0),
    ("prefill_z_misses_prompt_keys", "        zl[d] += fkp;\n      }\n      double dsum = 0.0;", "        zl[d] += 0.0 * fkp;\n      }\n      double dsum = 0.0;", 0),
]


def _mutate(src, old, new, occ):
    pos = -1
    for _ in range(occ + 1):
        pos = src.find(old, pos + 1)
        assert pos >= 0, f"mutation anchor not found: {old!r}"
    return src[:pos] + new + src[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, old, new, occ):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    c = tmp_path / "oracle_mut.c"
    c.write_text(mutated)
    lib = oracle.compile_c(str(c), str(tmp_path / "liboracle_mut.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ValueError) as e:
            failed.append(pin.__name__)
    assert failed, f"mutation {name} passed every pin"


# Slips in the Python part of the oracle (the projection in front of the
# decode step), planted in a copy of the method's source.
PY_MUTATIONS = [
    ("proj_k_and_v_swapped", "k = p[:, :, D:2 * D]", "k = p[:, :, 2 * D:3 * D]"),
    ("proj_columns_grouped_by_kind", "p = (x @ W).reshape(B, H, 2 * D + M)",
     "p = (x @ W).reshape(B, 2 * D + M, H).transpose(0, 2, 1)"),
    ("proj_w_transposed", "p = (x @ W).reshape(B, H, 2 * D + M)",
     "p = (x @ W.T.reshape(W.shape)).reshape(B, H, 2 * D + M)"),
]


@pytest.mark.parametrize("name,old,new", PY_MUTATIONS, ids=[m[0] for m in PY_MUTATIONS])
def test_pins_catch_projection_mutation(name, old, new):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.Oracle.decode_proj))
    assert src.count(old) == 1, f"mutation anchor not found: {old!r}"
    ns = dict(vars(oracle))
    exec(src.replace(old, new), ns)

    class Mutated(oracle.Oracle):
        decode_proj = ns["decode_proj"]

    orc = Mutated(oracle.default().path)
    with pytest.raises((AssertionError, ValueError)):
        P.pin_decode_proj(orc)
