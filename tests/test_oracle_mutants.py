"""Mistakes planted in a copy of the oracle must fail the oracle's pins.

Each mutant below is one plausible slip in one step of the oracle (a dropped term, a wrong
sign, index or bound, swapped operands or halves, a reversed tie order).  The test copies
oracle/ into a temporary directory, plants the mistake in the copy (the original is never
touched), compiles it, and runs the pin suites against the copy in a child process: the pins
must fail.  An unmodified copy must pass, which shows that the child really tests the copy.
Everything runs on the CPU; no GPU code is involved.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py")]
BUDGET_PINS = [os.path.join(ROOT, "tests", "test_budget_pins.py")]

C = "spin_oracle.c"
B = "budgets.py"
P = "oracle.py"

# (name, file, text in the oracle, planted replacement, pin suites)
MUTANTS = [
    # Philox4x64-10 (Salmon et al., SC'11) and the exploration draw layout
    ("philox-nine-rounds", C, "round < 10; ++round", "round < 9; ++round", PINS),
    ("philox-key-schedule", C, "k1 += PHILOX_W1;", "k1 += PHILOX_W0;", PINS),
    ("explore-key-halves-swapped", C,
     "(h & 1) ? (uint32_t)(w & 0xFFFFFFFFu) : (uint32_t)(w >> 32)",
     "(h & 1) ? (uint32_t)(w >> 32) : (uint32_t)(w & 0xFFFFFFFFu)", PINS),
    ("explore-counter-without-row", C,
     "uint64_t ctr[4] = {step, (uint64_t)(uint32_t)row,", "uint64_t ctr[4] = {step, (uint64_t)0,", PINS),
    # number formats
    ("e4m3-bias-8", C, "1.0 + (double)m / 8.0, e - 7)", "1.0 + (double)m / 8.0, e - 8)", PINS),
    ("e4m3-subnormal-scale", C, "ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)", PINS),
    ("bf16-low-half", C, "uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits;", PINS),
    # Algorithm 1's budget step and the exploration share of §3.2.1
    ("budget-floor-not-ceil", C, "* n_blocks + 9999) / 10000;", "* n_blocks) / 10000;", PINS),
    ("budget-topk-floor-truncated", C, "int64_t floor_k = (top_k + block - 1) / block;",
     "int64_t floor_k = top_k / block;", PINS),
    ("explore-count-uncapped", C, "return e < cap ? e : cap;", "return e;", PINS),
    # Eq. 1 and Eq. 2
    ("eq1-diagonal-off-by-one", C, "float d = D_req[q - i];", "float d = D_req[q - i + 1];", PINS),
    ("eq1-max-as-min", C,
     "float d = D_req[q - i];\n    if (cfg->combine == ORACLE_COMBINE_SUM) return v + d;\n    return v > d ? v : d;",
     "float d = D_req[q - i];\n    if (cfg->combine == ORACLE_COMBINE_SUM) return v + d;\n    return v < d ? v : d;",
     PINS),
    ("eq1-sum-as-difference", C,
     "float d = D_req[q - i];\n    if (cfg->combine == ORACLE_COMBINE_SUM) return v + d;",
     "float d = D_req[q - i];\n    if (cfg->combine == ORACLE_COMBINE_SUM) return v - d;", PINS),
    ("eq2-min-pooling", C, "if (p > s) s = p;", "if (p < s) s = p;", PINS),
    # §4.6 block-reduction ablations
    ("mean-divides-by-64", C, "return t[0] / (float)count;", "return t[0] / 64.0f;", PINS),
    ("top4-takes-three", C, "for (; c < 4; ++c) {", "for (; c < 3; ++c) {", PINS),
    ("a2-offset-sign", C, "float d = D_req[q / cfg->block - j];", "float d = D_req[q / cfg->block + j];",
     PINS),
    ("a2-observation-min", C, "if (!seen || z > zb) zb = z;", "if (!seen || z < zb) zb = z;", PINS),
    ("a0-without-forced-blocks", C,
     "        mask[0] = 1;\n        mask[nb - 1] = 1;\n        for (int64_t k = 0; k < cfg->top_k",
     "        for (int64_t k = 0; k < cfg->top_k", PINS),
    ("age-update-without-plus-one", C, "= (uint32_t)(step + 1);", "= (uint32_t)step;", PINS),
    # selection: forced blocks, warm-up, ranking, exploration, union
    ("newest-block-not-forced", C, "    mask[nb - 1] = 1;                                        /* newest",
     "    (void)0;                                                 /* newest", PINS),
    ("warm-up-ignored", C, "if (!warm) {", "if (0) {", PINS),
    ("ties-to-higher-index", C, "    return (x->j > y->j) - (x->j < y->j);\n}\n\nstatic int cmp_key_asc",
     "    return (x->j < y->j) - (x->j > y->j);\n}\n\nstatic int cmp_key_asc", PINS),
    ("explore-largest-keys", C, "if (x->u < y->u) return -1;\n    if (x->u > y->u) return 1;",
     "if (x->u < y->u) return 1;\n    if (x->u > y->u) return -1;", PINS),
    ("explore-among-selected", C, "if (!mask[j]) {\n                ex[ne].u",
     "if (1) {\n                ex[ne].u", PINS),
    ("union-of-row-zero-only", C, "if (mask[j]) { out[cnt++] = (int32_t)j; umask[j] = 1; }",
     "if (mask[j]) { out[cnt++] = (int32_t)j; if (r == 0) umask[j] = 1; }", PINS),
    # §2 indexer score
    ("score-without-relu", C, "z += wh * (x > 0.0 ? x : 0.0);", "z += wh * x;", PINS),
    ("score-without-fp8-scale", C, "double x = scale * dot;", "double x = dot;", PINS),
    ("score-scale-after-relu", C, "z += wh * (x > 0.0 ? x : 0.0);",
     "z += wh * scale * (dot > 0.0 ? dot : 0.0);", PINS),
    ("score-weight-of-head-zero", C, "double wh = (double)w_req[(int64_t)r * H + h];",
     "double wh = (double)w_req[(int64_t)r * H];", PINS),
    # Algorithm 1's top-K
    ("topk-counts-slots-past-n", C, "if (i >= n) continue;\n                    cand[nc].s",
     "cand[nc].s", PINS),
    # Algorithm 1's EMA update and the MTP replay of §3.2.2
    ("ema-weights-swapped", C, "float t = one_minus_alpha * z;\n                    V_req[i]",
     "float t = alpha * z;\n                    V_req[i]", PINS),
    ("replay-ignores-row-offset", C, "D_req[q + r - i] = fmaf(alpha, D_req[q + r - i], t);",
     "D_req[q - i] = fmaf(alpha, D_req[q - i], t);", PINS),
    ("replay-keeps-rejected-rows", C, "for (int64_t r = 0; r <= a; ++r) {", "for (int64_t r = 0; r < rows; ++r) {",
     PINS),
    ("explore-counter-per-block", C, "(uint64_t)(uint32_t)req, (uint64_t)(j >> 3)}",
     "(uint64_t)(uint32_t)req, (uint64_t)j}", PINS),
    ("e4m3-no-nan", C, "if (e == 0xF && m == 0x7) return NAN;", "", PINS),
    ("budget-not-capped-at-block-count", C, "return m < n_blocks ? m : n_blocks;", "return m;", PINS),
    ("explore-count-rounded", C, "int64_t e = ((int64_t)gamma_bp * m) / 10000;",
     "int64_t e = ((int64_t)gamma_bp * m + 5000) / 10000;", PINS),
    ("query-before-context-accepted", C, "if (n > 0 && q < n - 1) return 0;", "", PINS),
    ("scores-past-n-not-zero", C, "scores[o] = scored ? z[r] : 0.0f;", "scores[o] = scored ? z[r] : -1.0f;",
     PINS),
    ("topk-pads-with-zero", C, "out[k] = k < take ? sel[k] : -1;", "out[k] = k < take ? sel[k] : 0;", PINS),
    ("topk-in-score-order", C, "qsort(sel, (size_t)take, sizeof(int32_t), cmp_i32_asc);", "", PINS),
    ("replay-ignores-accepted", C, "int64_t a = accepted ? accepted[req] : 0;", "int64_t a = 0;", PINS),
    ("a2-update-at-slot-offset", C, "D_req[q / b - blk] = fmaf(alpha, D_req[q / b - blk], t);",
     "D_req[q - blk] = fmaf(alpha, D_req[q - blk], t);", PINS),
    ("reset-clears-every-request", C, "if (req >= 0 && r != req) continue;", "", PINS),
    ("philox-output-words-mixed", C, "uint64_t n1 = lo1;", "uint64_t n1 = lo0;", PINS),
    ("explore-key-without-layer", C, "uint64_t key[2] = {seed, (uint64_t)(uint32_t)layer};",
     "uint64_t key[2] = {seed, (uint64_t)0};", PINS),
    ("e4m3-unsigned", C, "return sign ? -v : v;", "return v;", PINS),
    ("budget-ignores-topk-floor", C, "int64_t m = floor_k > keep ? floor_k : keep;", "int64_t m = keep;", PINS),
    ("rho-override-ignored", C, "if (rho_bp < 0) rho_bp = cfg->rho_bp;", "", PINS),
    ("sink-block-not-forced", C, "    mask[0] = 1;                                             /* sink block */",
     "    (void)0;                                                 /* sink block */", PINS),
    ("mean-count-misses-last-slot", C, "for (int l = 0; l < 64; ++l) count += valid[l] != 0;",
     "for (int l = 0; l < 63; ++l) count += valid[l] != 0;", PINS),
    ("a0-one-slot-short", C, "for (int64_t k = 0; k < cfg->top_k && k < n_slots; ++k)",
     "for (int64_t k = 0; k < cfg->top_k - 1 && k < n_slots; ++k)", PINS),
    ("a0-without-dense-budget-rule", C, "if (oracle_budget(nb, cfg->top_k, b, rho_bp) >= nb) {", "if (0) {", PINS),
    ("a2-observation-counts-slots-past-n", C,
     "if (i >= n) continue;\n                    float z = scores[((int64_t)req * MB + k) * b + s];",
     "float z = scores[((int64_t)req * MB + k) * b + s];", PINS),
    ("score-slots-past-n", C, "int scored = valid_page && i < n;", "int scored = valid_page;", PINS),
    ("magnitude-signed", C, "adot += fabs(qv * kv);", "adot += qv * kv;", PINS),
    ("per-head-keys-as-shared", C, "int64_t kh = cfg->kv_heads == 1 ? 0 : h;", "int64_t kh = 0;", PINS),
    ("weights-of-request-zero", C, "const float* w_req = w + (int64_t)req * rows * H;", "const float* w_req = w;",
     PINS),
    ("query-of-request-zero", C, "const void* q_req = (const char*)q + (int64_t)req * q_elems * qsz;",
     "const void* q_req = (const char*)q;", PINS),
    ("topk-reads-row-zero", C, "cand[nc].s = scores[(((int64_t)req * rows + r) * MB + k) * b + s];",
     "cand[nc].s = scores[(((int64_t)req * rows) * MB + k) * b + s];", PINS),
    ("replay-reads-row-zero", C, "float z = scores[(((int64_t)req * rows + r) * MB + k) * b + s];",
     "float z = scores[(((int64_t)req * rows) * MB + k) * b + s];", PINS),
    ("reset-keeps-warm", C, "        warm[r] = 0;\n", "", PINS),
    # the whole step of one layer (select -> score -> top-K -> EMA, §3.2.2 for several rows)
    ("step-scores-row-zero-selection", P, "            blist, n_list = union, n_union",
     "            blist, n_list = blocks[:, 0, :], n_blocks[:, 0]", PINS),
    ("step-ignores-accepted", P,
     "ok4 = replay_ema(cfg, V, D, warm, scores, blist, n_list, n_slots, q_pos, rows, accepted)",
     "ok4 = replay_ema(cfg, V, D, warm, scores, blist, n_list, n_slots, q_pos, rows, None)", PINS),
    # per-layer budgets (project page, "Per-layer block budgets")
    ("miss-curve-without-forced", B, "chosen = set(forced) | set(free[: max(m - f, 0)])",
     "chosen = set(free[: max(m - f, 0)])", BUDGET_PINS),
    ("miss-curve-ties-to-higher-block", B, "key=lambda j: (-float(S[j]), j)", "key=lambda j: (-float(S[j]), -j)",
     BUDGET_PINS),
    ("allocate-spare-to-more-points", B, "(miss[l][g[l]], -g[l]) > (miss[best][g[best]], -g[best])",
     "(miss[l][g[l]], g[l]) > (miss[best][g[best]], g[best])", BUDGET_PINS),
    ("allocate-strict-miss-bound", B, "if miss[l][g] <= tau:", "if miss[l][g] < tau:", BUDGET_PINS),
    ("grid-point-as-sparsity", B, "return 10000 - g * 10000 // (n_points - 1)", "return g * 10000 // (n_points - 1)",
     BUDGET_PINS),
    ("miss-curve-kept-as-sparsity", B, "m = _o.budget(nb, top_k, 10000 - keep_bp)", "m = _o.budget(nb, top_k, keep_bp)",
     BUDGET_PINS),
    ("miss-curve-half-blocks", B, "missed = sum(1 for i in valid if i // 64 not in chosen)",
     "missed = sum(1 for i in valid if i // 32 not in chosen)", BUDGET_PINS),
    ("mean-curve-over-all-requests", B, "return [a / used for a in acc] if used else acc",
     "return [a / len(nbs) for a in acc] if used else acc", BUDGET_PINS),
    ("allocate-past-the-grid-top", B, "if g[l] >= G:", "if g[l] > G:", BUDGET_PINS),
    ("mean-curve-counts-empty-requests", B, "        if not any(int(i) >= 0 for i in topk):\n            continue\n",
     "", BUDGET_PINS),
]


def _copy(dst, mutant=None):
    os.makedirs(dst)
    for f in os.listdir(ORACLE_DIR):
        if f.endswith((".py", ".c", ".h")):
            shutil.copy(os.path.join(ORACLE_DIR, f), os.path.join(dst, f))
    if mutant is not None:
        _, fname, old, new, _ = mutant
        path = os.path.join(dst, fname)
        with open(path) as fh:
            text = fh.read()
        assert text.count(old) == 1, "mutant site must occur exactly once: %r" % old
        with open(path, "w") as fh:
            fh.write(text.replace(old, new))


def _run_pins(work, suites):
    """Builds the copy under work/oracle and runs the pin suites against it in a child whose
    import path puts the copy first.  Returns (exit code, output tail)."""
    src = os.path.join(work, "oracle", C)
    cc = subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o",
                         os.path.join(work, "oracle", "liboracle.so"), src, "-lm"],
                        capture_output=True, text=True)
    if cc.returncode != 0:
        return -1, cc.stderr[-2000:]
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([work, ROOT]), PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        *suites], cwd=work, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    base = tmp_path_factory.mktemp("oracle_mutants")
    jobs = {}
    for m in MUTANTS:
        _copy(os.path.join(str(base), m[0], "oracle"), m)
        jobs[m[0]] = (os.path.join(str(base), m[0]), m[4])
    _copy(os.path.join(str(base), "control", "oracle"))
    jobs["control"] = (os.path.join(str(base), "control"), PINS + BUDGET_PINS)
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = {name: ex.submit(_run_pins, work, suites) for name, (work, suites) in jobs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unmodified_copy_passes_its_pins(outcomes):
    rc, tail = outcomes["control"]
    assert rc == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(outcomes, name):
    rc, tail = outcomes[name]
    assert rc != -1, "the mutant did not compile:\n" + tail
    assert rc == 1, "the pins did not fail on the planted mistake (exit %d):\n%s" % (rc, tail)
