"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Every mutant is a textual edit of oracle.c (a dropped term, a wrong sign or
index, a transposed operand, a misread of the pages), compiled with gcc into a
throw-away library on the CPU.  The real oracle is never modified.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins

# name -> list of (old, new) replacements, each old string must occur in oracle.c
MUTANTS = {
    "diagonal kept": [("for (int j = i + 1; j < N; ++j) {\n                const float *vj",
                       "for (int j = i; j < N; ++j) {\n                if (j == i && i == 0) continue;\n                const float *vj")],
    "triangle before dense": [("memcpy(o, x, sizeof(float) * (size_t)D);", "memcpy(o + K, x, sizeof(float) * (size_t)D);"),
                              ("int64_t k = D + tri_pos(i, j, N);", "int64_t k = tri_pos(i, j, N);")],
    "column-major triangle": [("return i * N - i * (i + 1) / 2 + (j - i - 1);", "return j * (j - 1) / 2 + i + 0 * N;")],
    "dense vector last": [("return k == 0 ? dense + (size_t)b * D\n                  : pooled + ((size_t)b * T + (k - 1)) * D;",
                           "return k == T ? dense + (size_t)b * D\n                  : pooled + ((size_t)b * T + k) * D;")],
    "gram operand repeated": [("double p = (double)vi[d] * (double)vj[d];", "double p = (double)vi[d] * (double)vi[d];")],
    "mean not divided": [("                    v /= (double)L;\n", "")],
    "sum from +0.0": [("s[d] = started ? s[d] + v : v;", "s[d] = s[d] + v;")],
    "first lookup dropped": [("for (int64_t p = lo; p < hi; ++p) {\n                int64_t r = indices[p];\n                if (r < 0 || r >= num_rows[t]) {\n                    status |= ORACLE_INDEX_OOB;\n                    continue;\n                }\n                for",
                              "for (int64_t p = lo + (hi - lo > 1); p < hi; ++p) {\n                int64_t r = indices[p];\n                if (r < 0 || r >= num_rows[t]) {\n                    status |= ORACLE_INDEX_OOB;\n                    continue;\n                }\n                for")],
    "bf16 widened wrongly": [("(uint32_t)((const uint16_t *)table)[row * (int64_t)D + d] << 16", "(uint32_t)((const uint16_t *)table)[row * (int64_t)D + d] << 15")],
    "bwd drops upstream dx": [("dv[d] += (double)go[d];", "dv[d] += 0.0 * (double)go[d];")],
    "bwd wrong sign": [("dv[(size_t)i * D + d] += g * (double)vj[d];", "dv[(size_t)i * D + d] -= g * (double)vj[d];")],
    "bwd uses own row": [("dv[(size_t)i * D + d] += g * (double)vj[d];", "dv[(size_t)i * D + d] += g * (double)vec(dense, pooled, b, T, D, i)[d];")],
    "adagrad eps inside sqrt": [("double den = sqrt(A) + (double)eps;", "double den = sqrt(A + (double)eps);")],
    "adagrad sum not mean": [("double A = (double)accum[t][r] + ss / (double)D;", "double A = (double)accum[t][r] + ss;")],
    "adagrad uses old accumulator": [("double den = sqrt(A) + (double)eps;", "double den = sqrt((double)accum[t][r]) + (double)eps;")],
    "duplicates updated one by one": [("for (; e < n && refs[e].row == refs[s].row; ++e) {", "for (; e < n && e == s; ++e) {")],
    "bwd mean scale dropped": [("1.0 / (double)refs[e].L : 1.0;", "1.0 : 1.0;")],
    "sgd adds the gradient": [("w[d] = (float)((double)w[d] - (double)lr * g[d]);",
                               "w[d] = (float)((double)w[d] + (double)lr * g[d]);")],
    "sgd keeps the adagrad scale": [("w[d] = (float)((double)w[d] - (double)lr * g[d]);",
                                     "w[d] = (float)((double)w[d] - (double)lr * g[d] / (1.0 + sqrt(0.1)));")],
    "pooled gradient read from the wrong table": [("(size_t)(t + grad_t0) * D;", "(size_t)(T - 1 - t + grad_t0) * D;")],
    "hash as signed 64-bit": [("rows[p] = (int64_t)(raw[p] % (uint64_t)num_rows[t]);",
                               "rows[p] = (int64_t)raw[p] % num_rows[t];")],
    "hash with the next table's rows": [("rows[p] = (int64_t)(raw[p] % (uint64_t)num_rows[t]);",
                                         "rows[p] = (int64_t)(raw[p] % (uint64_t)num_rows[(t + 1) % T]);")],
    "oob lookup not counted": [("int64_t L = hi - lo;\n            int started = 0;",
                                "int64_t L = 0;\n            for (int64_t q = lo; q < hi; ++q) L += (indices[q] >= 0 && indices[q] < num_rows[t]);\n            int started = 0;")],
}


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, workdir):
    src = open(oracle.SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation site not found once: {old!r}"
        src = src.replace(old, new)
    tag = "".join(c if c.isalnum() else "_" for c in name)
    csrc = os.path.join(workdir, f"{tag}.c")
    lib = os.path.join(workdir, f"lib{tag}.so")
    with open(csrc, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", lib, csrc, "-lm"], check=True)
    orc = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the mutant '{name}'"
