"""The pins must catch a wrong oracle.

Each case plants one plausible mistake in a copy of the oracle's C source: a dropped term, a
wrong sign, an off-by-one index, a swapped operand or a reversed tie rule (none of them
writes outside its buffers). It builds that copy and runs every pin of test_oracle_pins.py,
test_oracle_fp8.py, test_oracle_int4.py and test_oracle_prefill.py against it, and at least
one pin must fail. The mistakes live only in the temporary copy; the oracle itself is
untouched.
"""
import inspect
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_fp8 as pins_fp8
import test_oracle_int4 as pins_int4
import test_oracle_pins as pins
import test_oracle_prefill as pins_prefill

# (name, text in dattn_oracle.c, replacement)
MUTATIONS = [
    ("logit without the scale",
     "        acc += orc_bf16_to_double(q[c]) * orc_bf16_to_double(k[c]);\n    return scale * acc;",
     "        acc += orc_bf16_to_double(q[c]) * orc_bf16_to_double(k[c]);\n    return acc;"),
    ("attention drops the last key",
     "    for (int64_t i = 0; i < n; ++i) e += exp(s[i] - m);\n    for (int64_t i = 0; i < n; ++i) {\n"
     "        const double w = exp(s[i] - m) / e;\n        const uint16_t *v",
     "    for (int64_t i = 0; i + 1 < n; ++i) e += exp(s[i] - m);\n    for (int64_t i = 0; i < n; ++i) {\n"
     "        const double w = exp(s[i] - m) / e;\n        const uint16_t *v"),
    ("partial weights with the wrong sign",
     "        const double w = exp(s[i] - m);\n        const uint16_t *v",
     "        const double w = exp(m - s[i]);\n        const uint16_t *v"),
    ("merge weights with the wrong sign", "            const double w = exp(m[j] - mg);",
     "            const double w = exp(mg - m[j]);"),
    ("merge forgets e_j", "            eg += e[j] * w;", "            eg += w;"),
    ("merged partial normalised twice", "        if (MA_g) MA_g[c] = acc[c];",
     "        if (MA_g) MA_g[c] = eg > 0.0 ? acc[c] / eg : 0.0;"),
    ("kv write one slot late", "        const int64_t slot = pos % P;",
     "        const int64_t slot = (pos + 1) % P;"),
    ("kv write does not count skipped tokens",
     "        if (page < 0 || page >= num_pages) { ++skipped; continue; }\n        const int64_t slot",
     "        if (page < 0 || page >= num_pages) { continue; }\n        const int64_t slot"),
    ("stats min uses max", "            if (bf16_to_float(k) < bf16_to_float(lo)) lo = k;",
     "            if (bf16_to_float(k) > bf16_to_float(lo)) lo = k;"),
    ("stats miss the last token of a page", "        for (int64_t t = t0 + 1; t < t1; ++t) {",
     "        for (int64_t t = t0 + 1; t + 1 < t1; ++t) {"),
    ("score ignores k_min", "        acc += a > b ? a : b;", "        acc += a;"),
    ("fp32 bound misses the factor d",
     "    return (double)d * ldexp(1.0, -23) * abs_sum + 2.0 * d * ldexp(1.0, -150);",
     "    return ldexp(1.0, -23) * abs_sum + 2.0 * d * ldexp(1.0, -150);"),
    ("fp32 bound sums signed terms", "        abs_sum += fabs(a > b ? a : b);",
     "        abs_sum += a > b ? a : b;"),
    ("physical bound keeps the last logical page", "                if (e > err) err = e;",
     "                err = e;"),
    ("physical score keeps the last logical page", "                if (s > best) best = s;",
     "                best = s;"),
    ("top-K ties go to the higher page",
     "            if (best < 0 || score[i] > score[best]) best = i; /* strict: lower index wins ties */",
     "            if (best < 0 || score[i] >= score[best]) best = i;"),
    ("top-K output not sorted", "        while (j >= 0 && sel[j] > v) { sel[j + 1] = sel[j]; --j; }",
     "        while (0) { sel[j + 1] = sel[j]; --j; }"),
    ("streaming window one token short", "        int64_t l0 = L - local;",
     "        int64_t l0 = L - local + 1;"),
    ("E4M3 rounds half away from zero", "    int n = (int)rint(a / ldexp(1.0, E - 3));",
     "    int n = (int)round(a / ldexp(1.0, E - 3));"),
    ("8-bit scale over 127 instead of 448", "    const float s = mx / 448.0f;",
     "    const float s = mx / 127.0f;"),
    ("8-bit write stores the V scale in the K scale pool",
     "            orc_quantize_row_fp8(v_new + src, d, v_pool + row * d, v_scale + row);",
     "            orc_quantize_row_fp8(v_new + src, d, v_pool + row * d, k_scale + row);"),
    ("4-bit scale over 8 instead of 7", "    const float s = mx / 7.0f;",
     "    const float s = mx / 8.0f;"),
    ("4-bit nibbles in the wrong order", "        packed[i] = (uint8_t)(nib[0] | (nib[1] << 4));",
     "        packed[i] = (uint8_t)(nib[1] | (nib[0] << 4));"),
    ("4-bit codes truncated instead of rounded",
     "                const float r = rintf(bf16_to_float(x[2 * i + j]) / s);",
     "                const float r = truncf(bf16_to_float(x[2 * i + j]) / s);"),
    ("4-bit codes rounded half away from zero",
     "                const float r = rintf(bf16_to_float(x[2 * i + j]) / s);",
     "                const float r = roundf(bf16_to_float(x[2 * i + j]) / s);"),
    ("4-bit decode with the wrong offset",
     "    return ((c & 1) ? (byte >> 4) : (byte & 15)) - 8;",
     "    return ((c & 1) ? (byte >> 4) : (byte & 15)) - 7;"),
    ("4-bit write stores the V scale in the K scale pool",
     "            orc_quantize_row_int4(v_new + src, d, v_pool + row * (d / 2), v_scale + row);",
     "            orc_quantize_row_int4(v_new + src, d, v_pool + row * (d / 2), k_scale + row);"),
    ("retrieval rows skip the partial last page",
     "            for (int64_t t = p * P; t < (p + 1) * P && t < L; ++t) rows[n++] = t;",
     "            if ((p + 1) * P > L) continue;\n"
     "            for (int64_t t = p * P; t < (p + 1) * P && t < L; ++t) rows[n++] = t;"),
    ("prefill band one block short", "            keep = kb < sink_blocks || kb > qb - local_blocks;",
     "            keep = kb < sink_blocks || kb > qb - local_blocks + 1;"),
    ("prefill ignores the causal bound", "    for (int64_t i = 0; i <= p; ++i) {",
     "    for (int64_t i = 0; i < L; ++i) {"),
    ("prefill query position off by one", "    const int64_t p = L - Tq + t;",
     "    const int64_t p = L - Tq + t - 1;"),
]


def _pin_calls():
    """Every pin of the oracle's pin modules as a list of zero-argument callables."""
    calls = []
    fns = inspect.getmembers(pins, inspect.isfunction) + \
        inspect.getmembers(pins_fp8, inspect.isfunction) + \
        inspect.getmembers(pins_int4, inspect.isfunction) + \
        inspect.getmembers(pins_prefill, inspect.isfunction)
    for name, fn in fns:
        if not name.startswith("test_"):
            continue
        params = list(inspect.signature(fn).parameters)
        marks = getattr(fn, "pytestmark", [])
        grids = [m.args for m in marks if m.name == "parametrize"]
        combos = [{}]
        for argnames, values in grids:
            names = [a.strip() for a in argnames.split(",")]
            new = []
            for c in combos:
                for v in values:
                    vv = v if len(names) > 1 else (v,)
                    new.append({**c, **dict(zip(names, vv))})
            combos = new
        for c in combos:
            kwargs = dict(c)
            if "orc" in params:
                kwargs["orc"] = oracle
            calls.append((f"{name}{c or ''}", lambda fn=fn, kw=kwargs: fn(**kw)))
    return calls


@pytest.fixture(scope="module")
def source():
    here = os.path.dirname(oracle.__file__)
    with open(os.path.join(here, "dattn_oracle.c")) as f:
        return f.read(), here


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(source, tmp_path, name, old, new):
    src, here = source
    assert src.count(old) == 1, f"the mutation anchor for '{name}' must occur exactly once"
    shutil.copy(os.path.join(here, "dattn_oracle.h"), tmp_path / "dattn_oracle.h")
    (tmp_path / "dattn_oracle.c").write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", *oracle.CFLAGS, str(tmp_path / "dattn_oracle.c"), "-o", lib_path,
                    "-lm"], check=True, cwd=tmp_path)
    mutant = oracle.load(lib_path)
    saved = oracle._lib
    oracle._lib = mutant  # the oracle's functions now call the mutant
    failed = []
    try:
        for label, call in _pin_calls():
            try:
                call()
            except AssertionError:
                failed.append(label)
    finally:
        oracle._lib = saved
    assert failed, f"no pin failed for the planted mistake: {name}"
