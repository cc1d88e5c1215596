"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of oracle/gdn_oracle.c (a flipped sign,
a dropped term, a wrong index or operand), builds that copy in a temporary
directory and runs tests/test_oracle_pins.py against it; at least one pin must
fail.  Every mutation keeps all memory accesses in bounds.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# name: (text in gdn_oracle.c, replacement)
MUTATIONS = {
    "delta_term_sign": ("double u = v[j] - alpha * sk;", "double u = v[j] + alpha * sk;"),
    "decay_dropped": ("row[i] = alpha * row[i] + beta * u * k[i];", "row[i] = row[i] + beta * u * k[i];"),
    "readout_uses_k": ("oj += row[i] * q[i];\n    o[j] = oj;\n  }\n}\n\n/* Features",
                       "oj += row[i] * k[i];\n    o[j] = oj;\n  }\n}\n\n/* Features"),
    "query_scale_missing": ("double qscale = 1.0 / sqrt((double)d->dk);", "double qscale = 1.0;"),
    "gqa_map_modulo": ("    int hq = h / G;\n    orc_delta_core", "    int hq = h % d->hk;\n    orc_delta_core"),
    "conv_taps_reversed": ("acc += conv_w[c * W + i] * hist[i * C + c];",
                           "acc += conv_w[c * W + (W - 2 - i)] * hist[i * C + c];"),
    "conv_history_not_appended": ("if (d->w > 1) memcpy(hist + (int64_t)(d->w - 2) * C, x",
                                  "if (0) memcpy(hist + (int64_t)(d->w - 2) * C, x"),
    "softplus_is_exp": ("return log1p(exp(x)); }", "return exp(x); }"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x)); }", "return 1.0 / (1.0 + exp(x)); }"),
    "norm_eps_missing": ("double r = 1.0 / sqrt(ss + ORC_EPS);", "double r = 1.0 / sqrt(ss);"),
    "alpha_is_g": ("f->alpha[h] = exp(f->g[h]);", "f->alpha[h] = f->g[h];"),
    "checkpoint_index": ("int64_t P = pos + 1;\n      if (P % ckpt_block) continue;\n      int64_t idx = P / ckpt_block - blk0 - 1;",
                         "int64_t P = pos + 1;\n      if (P % ckpt_block) continue;\n      int64_t idx = P / ckpt_block - blk0;"),
    "kda_checkpoint_after_next_token": ("int64_t P = p0 + (i - t0) + 1;", "int64_t P = p0 + (i - t0);"),
    "zero_keeps_conv": ("pool.conv[ids[i] * nc + e] = 0.0;", "pool.conv[ids[i] * nc + e] = 1.0;"),
    "commit_index_freed": ("if (t != L - 1) fr[k++] = sp[t];", "if (t != L - 1) fr[k++] = slot_ids[r];"),
    "pack_error_bit": ("if (c == 2 && err) *err |= ORC_ERR_SLOT_OOB;\n    for (int64_t e = 0; e < ns; ++e) st_ssm",
                       "if (c == 1 && err) *err |= ORC_ERR_SLOT_OOB;\n    for (int64_t e = 0; e < ns; ++e) st_ssm"),
    "chunk_state_decay_dropped": ("v += exp(blast - bcum[c]) * KR(c)[m] * Dm[c * dv + j];",
                                  "v += KR(c)[m] * Dm[c * dv + j];"),
    "chunk_gamma_sign": ("kk * exp(bcum[r] - bcum[c]);", "kk * exp(0.5 * (bcum[r] - bcum[c]));"),
    "kda_u_without_decay": ("sk += alpha[i] * row[i] * k[i];", "sk += row[i] * k[i];"),
    "kda_state_without_decay": ("row[i] = alpha[i] * row[i] + beta * u * k[i];",
                                "row[i] = row[i] + beta * u * k[i];"),
    "kda_window_kbar_decay": ("for (int64_t r = 0; r < nr; ++r) v += D[r] * KQ(r)[c] * exp(last - lb[r * dk + c]);",
                              "for (int64_t r = 0; r < nr; ++r) v += D[r] * KQ(r)[c] * exp(last);"),
    "rmsnorm_sum_not_mean": ("double inv = 1.0 / sqrt(ss / (double)dv + eps);",
                             "double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_gate_sigmoid": ("orc_silu(z[r * dv + j])", "orc_sigmoid(z[r * dv + j])"),
}


def _run_pins(name, tmp):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    d = os.path.join(tmp, name)
    os.makedirs(d, exist_ok=True)
    mutated = os.path.join(d, "gdn_oracle.c")
    with open(mutated, "w") as f:
        f.write(src.replace(old, new))
    env = dict(os.environ, GDN_ORACLE_SRC=mutated, GDN_ORACLE_BUILD_DIR=os.path.join(d, "build"),
               OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-600:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        res = dict(zip(MUTATIONS, ex.map(lambda n: _run_pins(n, tmp), MUTATIONS)))
    return res


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_fails_a_pin(outcomes, name):
    rc, tail = outcomes[name]
    # 1 = some pin failed (not 0 = all passed, not 2..5 = a collection or usage error)
    assert rc == 1, f"{name}: pytest exit {rc}\n{tail}"
