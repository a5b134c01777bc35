"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/oracle.cpp (a dropped term, a
wrong sign, a swapped index, a transposed operand), builds that copy on the
CPU, and runs the pin tests against it in a subprocess. The pins pass on the
real oracle, so each mutant must make at least one of them fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = [
    ("eps dropped", "mean_sq + eps", "mean_sq", "test_oracle_norm.py"),
    ("eps outside the root", "1.0 / std::sqrt(mean_sq + eps)", "1.0 / std::sqrt(mean_sq) + eps",
     "test_oracle_norm.py"),
    ("sum instead of mean", "sum_sq / static_cast<double>(D)", "sum_sq", "test_oracle_norm.py"),
    ("weight dropped", "x[j] * inv_rms * wj", "x[j] * inv_rms", "test_oracle_norm.py"),
    ("norm of the unrounded sum", "row[j] = load(x, r * x_row_stride + j, fmt);  // the rounded",
     "row[j] = sum;  // the rounded",
     "test_oracle_norm.py"),
    ("residual dropped", "load(x, r * x_row_stride + j, fmt) + load(res, r * res_row_stride + j, fmt)",
     "load(x, r * x_row_stride + j, fmt)", "test_oracle_norm.py"),
    ("rope first-half sign", "store(q, base + lo, xin[lo] * c - xin[hi] * sn, fmt);",
     "store(q, base + lo, xin[lo] * c + xin[hi] * sn, fmt);", "test_oracle_rope.py"),
    ("rope partner transposed", "store(q, base + hi, xin[hi] * c + xin[lo] * sn, fmt);",
     "store(q, base + hi, xin[lo] * c + xin[hi] * sn, fmt);", "test_oracle_rope.py"),
    ("K rotation skipped", "store(kv_cache, k_dst + lo, xin[lo] * c - xin[hi] * sn, fmt);",
     "store(kv_cache, k_dst + lo, xin[lo], fmt);", "test_oracle_rope.py"),
    ("interleaved partner as neox", "*hi = 2 * i + 1;", "*hi = i + h;", "test_oracle_rope.py"),
    ("cos and sin swapped", "const double c = c_row[i], sn = s_row[i];",
     "const double c = s_row[i], sn = c_row[i];", "test_oracle_rope.py"),
    ("K and V planes swapped", "(((0 * num_blocks + blk)", "(((1 * num_blocks + blk)",
     "test_oracle_rope.py"),
    ("slot offset from the quotient", "const int64_t off = sl % block_size;",
     "const int64_t off = sl / block_size % block_size;", "test_oracle_rope.py"),
    ("position bound off by one", "const bool pos_ok = p >= 0 && p < max_pos;",
     "const bool pos_ok = p >= 0 && p <= max_pos;", "test_oracle_rope.py"),
    ("gate and up swapped", "const double g = load(gate_up, t * in_row_stride + j, fmt);",
     "const double g = load(gate_up, t * in_row_stride + I + j, fmt);", "test_oracle_glu.py"),
    ("silu with e^+g", "a = g / (1.0 + std::exp(-g));", "a = g / (1.0 + std::exp(g));",
     "test_oracle_glu.py"),
    ("relu passes negatives", "a = g > 0.0 ? g : 0.0;", "a = g;", "test_oracle_glu.py"),
    ("uclip gamma dropped", "const float y = v * g;", "const float y = v;", "test_oracle_uclip.py"),
    ("uclip lower bound clips to the upper", "if (v < lo32) v = lo32;", "if (v < lo32) v = hi32;",
     "test_oracle_uclip.py"),
    ("uclip NaN passes the clamp", "if (std::isnan(v)) v = lo32;", "", "test_oracle_uclip.py"),
    ("uclip in double", "float v = a * xf;", "double v = static_cast<double>(a) * xf;", "test_oracle_uclip.py"),
    ("uclip alpha indexed by head", "alpha[alpha_per_channel ? d : 0]", "alpha[alpha_per_channel ? hh : 0]",
     "test_oracle_uclip.py"),
    ("uclip per-channel gamma read as scalar", "gamma[gamma_per_channel ? d : 0]", "gamma[0]",
     "test_oracle_uclip.py"),
    ("uclip middle stride ignored", "hh * x_h_stride + d", "hh * D + d", "test_oracle_uclip.py"),
    ("uclip gamma inside the clamp", "float v = a * xf;", "float v = a * g * xf;", "test_oracle_uclip.py"),
    ("attention without the max shift", "const double p = std::exp(s[t] - m);", "const double p = std::exp(s[t]);",
     "test_oracle_attention.py"),
    ("attention scale dropped", "s[t] = scale * dot;", "s[t] = dot;", "test_oracle_attention.py"),
    ("attention kv head by modulo", "static_cast<int64_t>(h / group) * head_dim", "static_cast<int64_t>(h % n_kv_head) * head_dim",
     "test_oracle_attention.py"),
    ("attention V read from the K plane", "load(kv_cache, v_plane + rows[t] + kvh_off + d, fmt)",
     "load(kv_cache, rows[t] + kvh_off + d, fmt)", "test_oracle_attention.py"),
    ("attention offset within the block dropped", "rows.push_back((blk * block_size + off)",
     "rows.push_back((blk * block_size)", "test_oracle_attention.py"),
    ("attention block table row ignored", "block_table[b * max_blocks + j]", "block_table[j]",
     "test_oracle_attention.py"),
    ("attention one token past seq_len", "j * block_size + off < L;", "j * block_size + off <= L;",
     "test_oracle_attention.py"),
    ("attention denominator dropped", "rows.empty() ? 0.0 : acc[d] / denom", "rows.empty() ? 0.0 : acc[d]",
     "test_oracle_attention.py"),
    ("linear weight transposed", "acc += hb[k] * load(W, n * K + k, fmt);", "acc += hb[k] * load(W, k * N + n, fmt);",
     "test_oracle_linear.py"),
    ("linear accumulates in float", "double acc = 0.0;\n            for (int64_t k = 0; k < K; ++k) acc += hb[k]",
     "float acc = 0.0f;\n            for (int64_t k = 0; k < K; ++k) acc += hb[k]", "test_oracle_linear.py"),
    ("ties away from zero", "(frac > 0.5 || (frac == 0.5 && std::fmod(fl, 2.0) != 0.0))",
     "(frac >= 0.5)", "test_oracle_rounding.py"),
    ("no overflow to infinity", "if (r > maxfin) r = INFINITY;", "", "test_oracle_rounding.py"),
]


@pytest.mark.parametrize("name,old,new,target", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, target):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    cpp = tmp_path / "oracle_mutant.cpp"
    so = tmp_path / "liboracle_mutant.so"
    cpp.write_text(mutated)
    subprocess.run(["g++", "-std=c++17", "-O1", "-ffp-contract=off", "-shared", "-fPIC",
                    "-o", str(so), str(cpp)], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", target)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
