"""The oracle's pins have teeth: each plausible mistake below, planted alone
in a copy of the oracle source (never in the file itself), compiled to a
separate library and loaded by a child pytest run of the pin tests, makes at
least one pin fail.  CPU only."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lamb1b_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py")]

# (what the mistake is, original text, mistaken text); each original occurs once
MUTATIONS = [
    ("c_bar's moving-average weights swapped",
     "fadd(fmul(s->cema, s->c_bar[l]), fmul(one_m_ema, c))",
     "fadd(fmul(one_m_ema, s->c_bar[l]), fmul(s->cema, c))"),
    ("c_bar starts at 1 instead of the first coefficient",
     "(s->n_warm == 0) ? c", "(s->n_warm == 0) ? 1.0f"),
    ("compression error with the wrong sign",
     "err[j] = pos ? fsub(z[j], s) : fadd(z[j], s);", "err[j] = pos ? fsub(s, z[j]) : fadd(z[j], s);"),
    ("chunk scale sqrt(S)/n instead of sqrt(S/n)",
     "float s = fsqrt(fdiv(S, (float)n));", "float s = fdiv(fsqrt(S), (float)n);"),
    ("tail chunk scaled by C instead of its element count",
     "float s = fsqrt(fdiv(S, (float)n));", "float s = fsqrt(fdiv(S, (float)C));"),
    ("server sum not divided by W",
     "float avg = fdiv(acc[j], (float)s->W);", "float avg = acc[j];"),
    ("server error not fed back",
     "z[j] = fadd(avg, s->e_s[base + j]);", "z[j] = avg;"),
    ("worker error not fed back",
     "z[j] = fadd(mw, ew[i]);", "z[j] = mw;"),
    ("layer factor not applied to the update",
     "s->c_cur[l] = fmul(s->c_bar[l], r);", "s->c_cur[l] = s->c_bar[l];"),
    ("soft threshold not relative to the previous factor",
     "float lo = fmul(fsub(1.0f, fthr), r_prev);", "float lo = fmul(fsub(1.0f, fthr), 1.0f);"),
    ("freeze starts the fresh variance at zero",
     "memcpy(s->v_fresh, s->v, (size_t)N * sizeof(float));",
     "memset(s->v_fresh, 0, (size_t)N * sizeof(float));"),
    ("per-tensor ratio as a minimum",
     "R = (rho[i] > R) ? rho[i] : R;", "R = (R == 0.0f || rho[i] < R) ? rho[i] : R;"),
    ("ratio inverted",
     "float r = fdiv(num, den);", "float r = fdiv(den, num);"),
    ("reconstructed gradient without the beta1 m_old term",
     "float gt = fdiv(fsub(m_new, fmul(s->beta1, s->m[i])), w1);", "float gt = fdiv(m_new, w1);"),
    ("fresh variance with beta2 and 1-beta2 swapped",
     "s->v_fresh[i] = fadd(fmul(s->beta2, s->v_fresh[i]), fmul(w2, fmul(gt, gt)));",
     "s->v_fresh[i] = fadd(fmul(w2, s->v_fresh[i]), fmul(s->beta2, fmul(gt, gt)));"),
    ("compression update preconditioned by the fresh variance",
     "    for (int64_t i = lo; i < hi; ++i) {\n        float d = fadd(fsqrt(s->v[i]), s->eps);\n        float u = fadd(fdiv(s->m[i], d), fmul(s->wd, s->x[i]));\n        s->x[i]",
     "    for (int64_t i = lo; i < hi; ++i) {\n        float d = fadd(fsqrt(s->v_fresh[i]), s->eps);\n        float u = fadd(fdiv(s->m[i], d), fmul(s->wd, s->x[i]));\n        s->x[i]"),
    ("no weight decay in the compression update",
     "        float u = fadd(fdiv(s->m[i], d), fmul(s->wd, s->x[i]));", "        float u = fdiv(s->m[i], d);"),
    ("zero-norm trust ratio 0 instead of 1",
     "(sx == 0.0f || su == 0.0f) ? 1.0f :", "(sx == 0.0f || su == 0.0f) ? 0.0f :"),
    ("trust ratio inverted",
     "fdiv(fsqrt(sx), fsqrt(su))", "fdiv(fsqrt(su), fsqrt(sx))"),
    ("warmup gradient summed, not averaged",
     "float gb = fdiv(acc, (float)s->W);", "float gb = acc;"),
    ("warmup second moment from m instead of the gradient",
     "s->v[i] = fadd(fmul(s->beta2, s->v[i]), fmul(w2, fmul(gb, gb)));",
     "s->v[i] = fadd(fmul(s->beta2, s->v[i]), fmul(w2, fmul(s->m[i], s->m[i])));"),
    ("sign of zero sent as -1",
     "int pos = !(z[j] < 0.0f);", "int pos = (z[j] > 0.0f);"),
    ("sign of NaN sent as -1 (zeros still +1)",
     "int pos = !(z[j] < 0.0f);", "int pos = (z[j] >= 0.0f);"),
    ("sign bits packed MSB first",
     "if (pos) words[j / 32] |= 1u << (j % 32);", "if (pos) words[j / 32] |= 1u << (31 - j % 32);"),
    ("1-bit Adam compression stage scaled by c_bar",
     "update_tensor(s, l, 1.0f);", "update_tensor(s, l, s->c_bar[l]);"),
    ("bfloat16 storage truncates instead of rounding to nearest even",
     "((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16)", "(b >> 16)"),
    ("1-bit Adam warmup applies LAMB's trust ratio",
     "        if (s->variant == 1) {\n            /* 1-bit Adam's warmup is vanilla Adam",
     "        if (s->variant == 99) {\n            /* 1-bit Adam's warmup is vanilla Adam"),
    ("server error kept unrounded under bfloat16 storage",
     "for (int64_t j = 0; j < n; ++j) s->e_s[base + j] = store_err(s, err[j]);",
     "for (int64_t j = 0; j < n; ++j) s->e_s[base + j] = err[j];"),
    ("sign words not cleared before packing",
     "for (int32_t q = 0; q < C / 32; ++q) words[q] = 0u;", ""),
    ("no weight decay in the warmup direction",
     "u[i] = fadd(fdiv(s->m[i], d), fmul(s->wd, s->x[i]));", "u[i] = fdiv(s->m[i], d);"),
    ("a NaN ratio ignored by the per-tensor maximum",
     "if (rho) rho[j] = (r != r) ? INFINITY : r;", "if (rho) rho[j] = r;"),
    ("worker momentum with beta1 and 1-beta1 swapped",
     "float mw = fadd(fmul(s->beta1, s->m[i]), fmul(w1, g[(int64_t)w * ld + i]));",
     "float mw = fadd(fmul(w1, s->m[i]), fmul(s->beta1, g[(int64_t)w * ld + i]));"),
    ("warmup momentum with beta1 and 1-beta1 swapped",
     "s->m[i] = fadd(fmul(s->beta1, s->m[i]), fmul(w1, gb));",
     "s->m[i] = fadd(fmul(w1, s->m[i]), fmul(s->beta1, gb));"),
    ("eps inside the square root of the warmup direction",
     "float d = fadd(fsqrt(s->v[i]), s->eps);\n        u[i] =",
     "float d = fsqrt(fadd(s->v[i], s->eps));\n        u[i] ="),
    ("trust ratio not clipped",
     "float c = clip(ratio, s->cmin, s->cmax);", "float c = ratio;"),
    ("compression-stage ratio not clipped to its factor bounds",
     "float r = clip(R, fmin, fmax);", "float r = R;"),
    ("scatter keeps each worker's own momentum (server result dropped)",
     "if (rho) rho[j] = (r != r) ? INFINITY : r;\n        s->m[i] = m_new;",
     "if (rho) rho[j] = (r != r) ? INFINITY : r;"),
    ("ratio taken from the fresh variance before this step's update",
     "s->v_fresh[i] = fadd(fmul(s->beta2, s->v_fresh[i]), fmul(w2, fmul(gt, gt)));\n"
     "        float num = fadd(fsqrt(s->v[i]), s->eps);\n"
     "        float den = fadd(fsqrt(s->v_fresh[i]), s->eps);",
     "float num = fadd(fsqrt(s->v[i]), s->eps);\n"
     "        float den = fadd(fsqrt(s->v_fresh[i]), s->eps);\n"
     "        s->v_fresh[i] = fadd(fmul(s->beta2, s->v_fresh[i]), fmul(w2, fmul(gt, gt)));"),
    ("compression-stage update without the learning rate",
     "float gc = fmul(s->lr, c);\n    for (int64_t i = lo; i < hi; ++i) {",
     "float gc = c;\n    for (int64_t i = lo; i < hi; ++i) {"),
    ("1-bit Adam tracks a fresh variance",
     "        if (s->variant == 1) {      /* 1-bit Adam: no fresh variance, no ratio */",
     "        if (s->variant == 99) {      /* 1-bit Adam: no fresh variance, no ratio */"),
]


@pytest.mark.parametrize("name,orig,mistake", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(name, orig, mistake, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, "the mutation no longer matches the oracle source"
    bad = tmp_path / "lamb1b_oracle_mutant.c"
    bad.write_text(src.replace(orig, mistake))
    so = tmp_path / "liblamb1b_oracle_mutant.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(bad), "-o", str(so), "-lm"])
    env = dict(os.environ, LAMB1B_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"no pin caught: {name}\n{r.stdout[-2000:]}"
