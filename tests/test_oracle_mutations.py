"""Plant plausible mistakes in copies of the oracle and check that a pin catches each.

Each mutation edits one line of oracle/gdn_oracle.c in a temporary copy (the
committed oracle is never touched), compiles it with gcc and reruns every pin
against it.  A mutation that no pin catches would mean the pins leave that part
of the oracle unchecked.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTATIONS = {
    "gqa_tiling": ("const int64_t hk = h / f;", "const int64_t hk = h % Hk;"),
    "no_decay": ("S[i * dv + j] = S[i * dv + j] * decay;", "S[i * dv + j] = S[i * dv + j];"),
    "conv_flipped": ("acc += w[d * K + j] * xv;", "acc += w[d * K + (K - 1 - j)] * xv;"),
    "delta_sign": ("delta[j] = b * (vt[j] - vpred[j]);", "delta[j] = b * (vt[j] + vpred[j]);"),
    "no_beta": ("delta[j] = b * (vt[j] - vpred[j]);", "delta[j] = (vt[j] - vpred[j]);"),
    "output_reads_key": ("acc += S[i * dv + j] * qt[i];", "acc += S[i * dv + j] * kt[i];"),
    "no_q_scale": ("qt[i] = qt[i] / s;", "qt[i] = qt[i];"),
    "no_k_norm": ("kt[i] = kt[i] / nk;", "kt[i] = kt[i];"),
    "silu_sign": ("y[d * L + t] = acc / (1.0 + exp(-acc));", "y[d * L + t] = acc / (1.0 + exp(acc));"),
    "conv_tail_off_by_one": ("int64_t p = P - (K - 1) + i;", "int64_t p = P - K + i;"),
    "update_transposed": ("S[i * dv + j] = S[i * dv + j] + kt[i] * delta[j];",
                          "S[i * dv + j] = S[i * dv + j] + kt[j % dk] * delta[i % dv];"),
    "eps_dropped": ("const double nq = sqrt(sq + eps), nk = sqrt(sk + eps);",
                    "const double nq = sqrt(sq), nk = sqrt(sk);"),
    "v_from_key_head": ("vt[j] = y[(v0 + h * dv + j) * L + t];", "vt[j] = y[(v0 + hk * dv + j) * L + t];"),
    "gate_sign": ("gate[t * H + h] = -exp(A_log[h]) * sp;", "gate[t * H + h] = exp(A_log[h]) * sp;"),
    "gate_no_dt_bias": ("const double x = a[t * H + h] + dt_bias[h];", "const double x = a[t * H + h];"),
    "softplus_as_relu": ("const double sp = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));",
                         "const double sp = (x > 0.0 ? x : 0.0);"),
    "beta_sign": ("beta[t * H + h] = 1.0 / (1.0 + exp(-b[t * H + h]));",
                  "beta[t * H + h] = 1.0 / (1.0 + exp(b[t * H + h]));"),
    "rmsnorm_sum_not_mean": ("const double rms = sqrt(sq / (double)n + eps);", "const double rms = sqrt(sq + eps);"),
    "rmsnorm_no_eps": ("const double rms = sqrt(sq / (double)n + eps);", "const double rms = sqrt(sq / (double)n);"),
    "rmsnorm_gate_sign": ("(zz / (1.0 + exp(-zz)))", "(zz / (1.0 + exp(zz)))"),
    "rmsnorm_no_weight": ("y[r * n + j] = weight[j] * (o[r * n + j] / rms)", "y[r * n + j] = (o[r * n + j] / rms)"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path, oracle_mod):
    old, new = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old}"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / "libmut.so"))
    caught = []
    with oracle.use_library(lib):
        for pin in ALL_PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin.__name__)
    assert caught, f"mutation {name} passed every pin"
