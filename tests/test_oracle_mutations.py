"""The pins must catch plausible mistakes in the oracle.

Each case below plants one mistake in a copy of oracle.c (compiled on the CPU
into a temporary directory) and runs every pin of test_oracle_pins.py against
that copy; at least one pin has to fail. The real oracle is never modified.
"""
import inspect

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTATIONS = {
    "readout_before_update": (
        """        for (int64_t n = 0; n < N; ++n) {
            double dA = exp(dl * (double)A[d * N + n]);   /* deltaA */
            double dB = dl * (double)B[bt * N + n];        /* deltaB */
            if (zoh)
                dB *= zoh_factor(dl * (double)A[d * N + n]);
            h[n] = dA * h[n] + dB * xv;
        }
        for (int64_t n = 0; n < N; ++n)
            acc += h[n] * (double)C[bt * N + n];
""",
        """        for (int64_t n = 0; n < N; ++n)
            acc += h[n] * (double)C[bt * N + n];
        for (int64_t n = 0; n < N; ++n) {
            double dA = exp(dl * (double)A[d * N + n]);   /* deltaA */
            double dB = dl * (double)B[bt * N + n];        /* deltaB */
            if (zoh)
                dB *= zoh_factor(dl * (double)A[d * N + n]);
            h[n] = dA * h[n] + dB * xv;
        }
"""),
    "exp_sign": ("double dA = exp(dl * (double)A[d * N + n]);   /* deltaA */",
                 "double dA = exp(-dl * (double)A[d * N + n]);   /* deltaA */"),
    "A_transposed": ("double dA = exp(dl * (double)A[d * N + n]);   /* deltaA */",
                     "double dA = exp(dl * (double)A[n * D + d]);   /* deltaA */"),
    "dropped_input_term": ("            h[n] = dA * h[n] + dB * xv;\n        }\n        for",
                           "            h[n] = dA * h[n];\n        }\n        for"),
    "deltaB_without_delta": ("double dB = dl * (double)B[bt * N + n];        /* deltaB */",
                             "double dB = (double)B[bt * N + n];        /* deltaB */"),
    "B_ignores_time": ("double dB = dl * (double)B[bt * N + n];        /* deltaB */",
                       "double dB = dl * (double)B[b * L * N + n];        /* deltaB */"),
    "C_previous_step": ("            acc += h[n] * (double)C[bt * N + n];\n        if (y_out)",
                        "            acc += h[n] * (double)C[(t > 0 ? bt - 1 : bt) * N + n];\n        if (y_out)"),
    "x_wrong_channel": ("double xv = (double)x[bt * D + d];",
                        "double xv = (double)x[bt * D + (D - 1 - d)];"),
    "h0_ignored": ("h[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;", "h[n] = 0.0;"),
    "hT_not_written": ("            h_out[n] = h[n];", "            h_out[n] = 0.0;"),
    "softplus_missing_max_term": ("return (u > 0.0 ? u : 0.0) + log1p(exp(-a));",
                                  "return log1p(exp(-a));"),
    "softplus_flag_ignored": ("        if (delta_softplus)\n            dl = oracle_softplus(dl);\n", ""),
    "step_wrong_decay": ("            double dA = exp(dl * (double)A[d * N + n]);\n            double dB = dl * (double)B[b * N + n];",
                         "            double dA = exp(dl * (double)A[n]);\n            double dB = dl * (double)B[b * N + n];"),
    "gate_sign": ("y *= zv / (1.0 + exp(-zv));", "y *= zv / (1.0 + exp(zv));"),
    "gate_without_z": ("y *= zv / (1.0 + exp(-zv));", "y *= 1.0 / (1.0 + exp(-zv));"),
    "skip_dropped": ("        y += (double)Dskip[d] * xv;\n", ""),
    "skip_wrong_channel": ("y += (double)Dskip[d] * xv;", "y += (double)Dskip[0] * xv;"),
    "skip_after_gate": ("""    if (Dskip)
        y += (double)Dskip[d] * xv;
    if (z) {
        double zv = (double)z[btd];
        y *= zv / (1.0 + exp(-zv));
    }""", """    if (z) {
        double zv = (double)z[btd];
        y *= zv / (1.0 + exp(-zv));
    }
    if (Dskip)
        y += (double)Dskip[d] * xv;"""),
    "zoh_without_division": ("return w == 0.0 ? 1.0 : expm1(w) / w;", "return w == 0.0 ? 1.0 : expm1(w);"),
    "zoh_uses_exp": ("return w == 0.0 ? 1.0 : expm1(w) / w;", "return w == 0.0 ? 1.0 : exp(w) / w;"),
    "zoh_flag_ignored": ("            if (zoh)\n                dB *= zoh_factor(dl * (double)A[d * N + n]);\n", ""),
    "conv_taps_reversed": ("acc += (double)w[d * K + k] * v;", "acc += (double)w[d * K + (K - 1 - k)] * v;"),
    "conv_bias_dropped": ("double acc = bias ? (double)bias[d] : 0.0;", "double acc = 0.0;"),
    "conv_shift_off_by_one": ("int64_t tau = t - (K - 1) + k;", "int64_t tau = t - K + k;"),
    "conv_state_newest_first": ("v = state_in ? (double)state_in[(b * D + d) * (K - 1) + (K - 1 + tau)] : 0.0;",
                                "v = state_in ? (double)state_in[(b * D + d) * (K - 1) + (-1 - tau)] : 0.0;"),
    "step_dropped_input": ("            h[n] = dA * h[n] + dB * xv;\n        }\n        for (int64_t n = 0; n < N; ++n)\n            acc += h[n] * (double)C[b * N + n];",
                           "            h[n] = dA * h[n];\n        }\n        for (int64_t n = 0; n < N; ++n)\n            acc += h[n] * (double)C[b * N + n];"),
    "bwd_sigmoid_dropped": ("                    gdl *= 1.0 / (1.0 + exp(-u));", ""),
    "bwd_dC_previous_state": ("dC[bt * N + n] += gyv * hs[(t + 1) * N + n];",
                              "dC[bt * N + n] += gyv * hs[t * N + n];"),
    "bwd_no_decay_carry": ("                    g[n] *= a;                                      /* into h_{t-1} */\n", ""),
    "bwd_dA_without_dl": ("dA[d * N + n] += da * a * dl;", "dA[d * N + n] += da * a;"),
    "bwd_dx_without_dl": ("gx += g[n] * dl * Bn;", "gx += g[n] * Bn;"),
    "bwd_ddelta_drops_decay_term": ("gdl += da * a * an + g[n] * Bn * xv;", "gdl += g[n] * Bn * xv;"),
    "bwd_dh0_before_last_decay": ("        for (int64_t n = 0; n < N; ++n)\n                    dh0[(b * D + d) * N + n] = g[n];",
                                  "        for (int64_t n = 0; n < N; ++n)\n                    dh0[(b * D + d) * N + n] = g[n] / exp(dls[0] * (double)A[d * N + n]);"),
    "bwd_ghT_ignored": ("g[n] = ghT ? ghT[(b * D + d) * N + n] : 0.0;", "g[n] = 0.0;"),
    "ssd_decay_first_head": ("const double a = exp(dl * (double)A[hd]);", "const double a = exp(dl * (double)A[0]);"),
    "ssd_input_without_dt": ("const double db = dl * (double)B[bt * N + n];", "const double db = (double)B[bt * N + n];"),
    "ssd_readout_uses_B": ("acc += (double)C[bt * N + n] * h[n * P + p];", "acc += (double)B[bt * N + n] * h[n * P + p];"),
    "ssd_h0_ignored": ("h[i] = h0 ? h0[s0 + i] : 0.0;", "h[i] = 0.0;"),
    "ssd_x_first_column": ("h[n * P + p] = a * h[n * P + p] + db * (double)xv[p];",
                           "h[n * P + p] = a * h[n * P + p] + db * (double)xv[0];"),
    "ssd_softplus_ignored": ("                if (dt_softplus)\n                    dl = oracle_softplus(dl);\n                const double a", "                const double a"),
    "bwd_gate_derivative_partial": ("dz[i] = dout[i] * pre * s * (1.0 + zv * (1.0 - s));", "dz[i] = dout[i] * pre * s;"),
    "bwd_gate_scan_gradient_ungated": ("                g *= zv / (1.0 + exp(-zv));\n", ""),
    "bwd_skip_missing_from_dx": ("                dx[i] += gy[i] * (double)Dskip[d];\n", ""),
    "bwd_dDskip_ungated": ("dDskip[d] += gy[i] * xv;", "dDskip[d] += dout[i] * xv;"),
    "bwd_dz_without_skip": ("const double pre = y[i] + (Dskip ? (double)Dskip[d] * xv : 0.0);", "const double pre = y[i];"),
}


def _pin_calls():
    """(name, callable(orc)) for every pin, expanding parametrized ones."""
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            out.append((name, lambda o, fn=fn: fn(o)))
            continue
        (argnames, values), = [m.args for m in marks]
        argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for v in values:
            v = v if isinstance(v, tuple) and len(argnames) > 1 else (v,)
            kw = dict(zip(argnames, v))
            out.append((f"{name}{v}", lambda o, fn=fn, kw=kw: fn(o, **kw)))
    return out


def test_unmutated_copy_passes_every_pin(tmp_path):
    src = open(oracle.SRC).read()
    p = tmp_path / "same.c"
    p.write_text(src)
    o = oracle.compile_variant(str(p), str(tmp_path / "same.so"))
    for name, call in _pin_calls():
        call(o)


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_mutation_is_caught(tmp_path, mutation):
    old, new = MUTATIONS[mutation]
    src = open(oracle.SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {mutation} not found"
    p = tmp_path / f"{mutation}.c"
    p.write_text(src.replace(old, new, 1))
    o = oracle.compile_variant(str(p), str(tmp_path / f"{mutation}.so"))
    failed = []
    for name, call in _pin_calls():
        try:
            call(o)
        except (AssertionError, RuntimeError):
            failed.append(name)
    assert failed, f"no pin caught the planted mistake '{mutation}'"
