"""The pins reject a plausibly broken oracle (CPU only).

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign or bound, a wrong index, a swapped operand), compiles the
copy to a temporary library and runs the pin suite against it in a child
process: the pins must fail.  The committed oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

MUTATIONS = {
    "sink scaled by sm_scale": (
        "const double sink = J->sink ? (double)J->sink[h] : -INFINITY;",
        "const double sink = J->sink ? (double)J->sink[h] * J->sm_scale : -INFINITY;"),
    "sink dropped from the denominator": (
        "double z = exp(sink - m);", "double z = 0.0 * exp(sink - m);"),
    "window bound off by one": (
        "qpos - J->window_left <= (int64_t)j", "qpos - J->window_left < (int64_t)j"),
    "causal bound off by one": (
        "(int64_t)j <= qpos", "(int64_t)j < qpos"),
    "causal flag ignored": (
        "if (J->causal && !((int64_t)j <= qpos)) allowed = 0;",
        "if (!((int64_t)j <= qpos)) allowed = 0;"),
    "GQA head mapping modulo": (
        "const int g = h / group;", "const int g = h % Hkv;"),
    "causal mask aligned to the start": (
        "const int64_t qpos = (int64_t)kv_len - q_len + i_row;",
        "const int64_t qpos = (int64_t)i_row;"),
    "page offset dropped from the slot": (
        "return (int64_t)page * block_size + pos % block_size;",
        "return (int64_t)page * block_size;"),
    "values read from the key pool": (
        "o[d] += p * widen(J->v_cache, J->kv_dtype, vbase + d);",
        "o[d] += p * widen(J->k_cache, J->kv_dtype, vbase + d);"),
    "sm_scale dropped": (
        "s_buf[j] = J->sm_scale * dot;", "s_buf[j] = dot;"),
    "request bound inclusive": (
        "if (cu[r] <= t && t < cu[r + 1]) {", "if (cu[r] <= t && t <= cu[r + 1]) {"),
    "rope: sine term with the wrong sign": (
        "out[row + a] = xa * c - xb * s;", "out[row + a] = xa * c + xb * s;"),
    "rope: frequency exponent without the 2": (
        "pow(base, -2.0 * i / rotary_dim)", "pow(base, -1.0 * i / rotary_dim)"),
    "rope: neox pairs off by one": (
        "const int b = neox ? i + half : 2 * i + 1;",
        "const int b = neox ? i + half - 1 : 2 * i + 1;"),
    "rope: position scale multiplies": (
        "(double)positions[t] / position_scale", "(double)positions[t] * position_scale"),
    "rope: NTK exponent inverted": (
        "pow(ntk_alpha, (double)rotary_dim / (rotary_dim - 2))",
        "pow(ntk_alpha, (double)(rotary_dim - 2) / rotary_dim)"),
    "rope: unrotated tail dropped": (
        "for (int d = 0; d < head_dim; ++d) out[row + d] = widen(x, dtype, row + d);",
        "for (int d = 0; d < head_dim; ++d) out[row + d] = 0.0;"),
    "alibi: distance with the wrong sign": (
        "(double)J->alibi[h] * (double)((int64_t)j - qpos)",
        "(double)J->alibi[h] * (double)(qpos - (int64_t)j)"),
    "alibi: slope of the kv head": (
        "(double)J->alibi[h] * (double)((int64_t)j - qpos)",
        "(double)J->alibi[h / group] * (double)((int64_t)j - qpos)"),
    "alibi: bias scaled by sm_scale": (
        "if (J->alibi) s_buf[j] += (double)J->alibi[h]",
        "if (J->alibi) s_buf[j] += J->sm_scale * (double)J->alibi[h]"),
    "minference: slash summed per key, not per diagonal": (
        "sh[pos - j] += p;", "sh[j] += p;"),
    "minference: estimating queries taken from the start": (
        "const int pos = S - last_q + i;", "const int pos = i;"),
    "sparse attention: vertical and slash intersected": (
        "if (!(isv[j] || iss[i - j]))", "if (!(isv[j] && iss[i - j]))"),
    "cache write ignores the skip marker": (
        "if (s < 0) continue;", "if (s < -1) continue;"),
    "lse in log2 units": (
        "J->lse[(int64_t)out_row * Hq + h] = m + log(z);",
        "J->lse[(int64_t)out_row * Hq + h] = m + log2(z);"),
    "lse without the row maximum": (
        "J->lse[(int64_t)out_row * Hq + h] = m + log(z);",
        "J->lse[(int64_t)out_row * Hq + h] = log(z);"),
    "minference: estimate softmax not normalised": (
        "const double p = exp(s[j] - m) / z;\n                vh[j] += p;",
        "const double p = exp(s[j] - m);\n                vh[j] += p;"),
    "minference: estimate ignores the scale": (
        "for (int j = 0; j <= pos; ++j) {\n                const int64_t kb = ((int64_t)j * Hkv + kvh) * D;\n"
        "                double dot = 0.0;\n"
        "                for (int d = 0; d < D; ++d) dot += widen(q, dtype, qb + d) * widen(k, dtype, kb + d);\n"
        "                s[j] = scale * dot;",
        "for (int j = 0; j <= pos; ++j) {\n                const int64_t kb = ((int64_t)j * Hkv + kvh) * D;\n"
        "                double dot = 0.0;\n"
        "                for (int d = 0; d < D; ++d) dot += widen(q, dtype, qb + d) * widen(k, dtype, kb + d);\n"
        "                s[j] = dot;"),
    "sparse attention: diagonal indexed by the key": (
        "if (!(isv[j] || iss[i - j]))", "if (!(isv[j] || iss[j]))"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-fPIC",
                    "-shared", "-pthread", str(mut), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins accepted the mutant '{name}':\n{r.stdout[-2000:]}"
