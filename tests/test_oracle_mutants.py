"""Each plausible mistake, planted in a copy of the oracle on the CPU, must
fail at least one pin.  This checks that the pins constrain every term of
the oracle, not only that the oracle passes them."""
import os
import shutil

import pytest

import oracle
import oracle_pins

# (name, text in ssm_oracle.c, replacement) -- every mutant stays in bounds.
MUTANTS = [
    ("drop_delta_in_input_term", "if (!zoh) return dt;", "if (!zoh) return 1.0;"),
    ("zoh_sign", "expm1(dt * a) / a", "expm1(-dt * a) / a"),
    ("zoh_no_divide", "expm1(dt * a) / a", "expm1(dt * a)"),
    ("zoh_limit_at_zero", "expm1(dt * a) / a : dt;", "expm1(dt * a) / a : 0.0;"),
    ("zoh_ignored", "return a != 0.0 ? expm1(dt * a) / a : dt;", "return dt;"),
    ("h0_ignored", "h[n] = j->h0 ? j->h0[k * N + n] : 0.0;", "h[n] = 0.0;"),
    ("conv_taps_reversed", "acc += load(pio, w, d * K + k) * xv;", "acc += load(pio, w, d * K + (K - 1 - k)) * xv;"),
    ("conv_off_by_one", "const int64_t src = t - (K - 1) + k;", "const int64_t src = t - K + k;"),
    ("conv_bias_ignored", "double acc = cbias ? load(pio, cbias, d) : 0.0;", "double acc = 0.0;"),
    ("conv_no_silu", "u[c * seqlen + t] = silu(acc);", "u[c * seqlen + t] = acc;"),
    ("conv_state_ignored", "else if (state)", "else if (0)"),
    ("wrong_sign_in_decay", "exp(dt * a) * h[n]", "exp(-dt * a) * h[n]"),
    ("drop_skip_term", "yv += Dskip * x;", "(void)Dskip;"),
    ("gate_sigmoid_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("softplus_wrong", "return log1p(exp(v));", "return exp(v);"),
    ("C_replaced_by_B", "yv += load(j->io, j->C, bc_row", "yv += load(j->io, j->B, bc_row"),
    ("A_transposed", "load(j->pio, j->A, d * N + n)", "load(j->pio, j->A, n * j->dim + d)"),
    ("B_ignores_batch", "const int64_t bc_row = b * L * N;", "const int64_t bc_row = 0 * b;"),
    ("bias_ignored", "+ bias;\n        const double dt", ";\n        const double dt"),
    ("state_not_reset", "h[n] = j->h0 ? j->h0[k * N + n] : 0.0;", "if (j->h0) h[n] = j->h0[k * N + n];"),
    ("gate_on_state_only", "yv += Dskip * x;\n        if (j->z) yv *= silu(load(j->io, j->z, row + t));",
     "if (j->z) yv *= silu(load(j->io, j->z, row + t));\n        yv += Dskip * x;"),
    ("step_skips_softplus", "const double dt = delta_softplus ? softplus(v) : v;", "const double dt = v;"),
    ("step_state_index", "double* h = state + c * dstate;", "double* h = state + d * dstate;"),
    ("output_before_update", None, None),  # built below: y read from the previous state
]


def _output_before_update(src):
    upd = ("        for (int64_t n = 0; n < N; n++) {\n"
           "            const double a = load(j->pio, j->A, d * N + n);\n"
           "            const double Bv = load(j->io, j->B, bc_row + t * N + n);\n"
           "            h[n] = exp(dt * a) * h[n] + input_weight(j->zoh, dt, a) * Bv * x;\n"
           "        }\n")
    out = ("        for (int64_t n = 0; n < N; n++)\n"
           "            yv += load(j->io, j->C, bc_row + t * N + n) * h[n];\n")
    assert upd in src and out in src
    return src.replace(upd + out, out + upd)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    if name == "output_before_update":
        mutated = _output_before_update(src)
    else:
        assert old in src, f"mutation site for {name} not found"
        mutated = src.replace(old, new)
    assert mutated != src
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = oracle.load(oracle.build(path, os.path.join(tmp_path, f"libmut_{name}.so")))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
