"""Planted mistakes in the oracle must fail its pins (CPU only).

Each entry of ``MUTANTS`` copies the oracle's C source, turns one expression
into a plausible slip (a dropped term, a flipped comparison, a row or index
off by one, a swapped operand), builds the copy with the oracle's compiler
flags, and runs ``tests/test_oracle_pins.py`` against it in a child process.
The child must end with failed tests (pytest exit status 1); the first pin
that failed is named in the report.  An unchanged copy, built and run the
same way, must pass every pin: that shows the failures come from the slips
and not from the harness.  The copies live in a temporary directory; the
oracle's own source and build are never touched.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "d3d_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")
# the oracle's own flags (oracle.build): IEEE arithmetic, no contraction
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]

# (name, expression in the oracle, the slip); each expression occurs once.
MUTANTS = [
    # bf16 decoding and the segment-table checks
    ("bf16_shift", "((uint32_t)b) << 16", "((uint32_t)b) << 15"),
    ("segments_parent_may_be_bidir", "if (pg[2] != OR_CAUSAL || pg[3] != -1)", "if (pg[3] != -1)"),
    ("segments_allow_gap", "if (g[0] != next || g[1] < 1)", "if (g[0] < next || g[1] < 1)"),
    # packed drafting attention: visibility, scale, softmax, GQA map, dense mask
    ("causal_excludes_diagonal", "g[2] == OR_BIDIR ? 1 : (j <= i)", "g[2] == OR_BIDIR ? 1 : (j < i)"),
    ("block_never_bidirectional", "g[2] == OR_BIDIR ? 1 : (j <= i)", "(j <= i)"),
    ("parent_overreach", "if (j >= pg[0] && j < pg[0] + g[4])", "if (j >= pg[0] && j <= pg[0] + g[4])"),
    ("scale_dropped", "score[k] = scale * acc;", "score[k] = acc;"),
    ("softmax_unnormalised", "double w = score[k] / z;", "double w = score[k];"),
    ("gqa_head_modulo", "                int hk = h / G;\n                int nk = 0;",
     "                int hk = h % Hkv;\n                int nk = 0;"),
    ("dense_mask_no_diagonal", "int own_hi = (g[2] == OR_BIDIR) ? len : a + 1;",
     "int own_hi = (g[2] == OR_BIDIR) ? len : a;"),
    # speculative-sampling verification
    ("temperature_multiplies", "p[v] = logit_value(base, dtype, off + v) / T;",
     "p[v] = logit_value(base, dtype, off + v) * T;"),
    ("alpha_inverted", "al[j] = (pj >= qj) ? 1.0 : pj / qj;", "al[j] = (pj >= qj) ? 1.0 : qj / pj;"),
    ("alpha_unclamped", "al[j] = (pj >= qj) ? 1.0 : pj / qj;", "al[j] = pj / qj;"),
    ("accept_if_u_above", "if (u < al[a])", "if (u > al[a])"),
    ("residual_q_minus_p", "res[v] = (P[v] > Q[v]) ? P[v] - Q[v] : 0.0;",
     "res[v] = (Q[v] > P[v]) ? Q[v] - P[v] : 0.0;"),
    ("residual_is_target", "res[v] = (P[v] > Q[v]) ? P[v] - Q[v] : 0.0;", "res[v] = P[v];"),
    ("cdf_target_not_scaled", "double target = u * S, c = 0.0;", "double target = u, c = 0.0;"),
    ("margin_sample_unnormalised", "*margin = (lo < hi ? lo : hi) / S;", "*margin = (lo < hi ? lo : hi);"),
    ("margin_sample_far_end", "*margin = (lo < hi ? lo : hi) / S;", "*margin = (lo > hi ? lo : hi) / S;"),
    ("margin_accept_last_test_only", "if (gap < mA)\n                mA = gap;", "mA = gap;"),
    ("fallback_not_recorded", "fb = 1;\n                t = inverse_cdf(P,", "fb = 0;\n                t = inverse_cdf(P,"),
    ("fallback_never_fires", "if (t < 0) {\n                fb = 1;", "if (t < -1) {\n                fb = 1;"),
    ("bonus_from_wrong_row", "softmax_row(target, dtype, ((size_t)r * B + (B - 1)) * V, V, T, P);",
     "softmax_row(target, dtype, ((size_t)r * B + (B - 2)) * V, V, T, P);"),
    ("resample_from_next_row", "softmax_row(target, dtype, ((size_t)r * B + a) * V, V, T, P);",
     "softmax_row(target, dtype, ((size_t)r * B + a + 1) * V, V, T, P);"),
    ("num_tokens_without_the_extra_token",
     "num_tokens[r] = a + 1;\n        for (int j = 0; j < B; ++j) {\n            int32_t tok = -1;",
     "num_tokens[r] = a;\n        for (int j = 0; j < B; ++j) {\n            int32_t tok = -1;"),
    # AWL weights
    ("awl_includes_own_position", "            w[(size_t)r * Bm1 + k] = prod;\n            prod *= alpha[(size_t)r * Bm1 + k];",
     "            prod *= alpha[(size_t)r * Bm1 + k];\n            w[(size_t)r * Bm1 + k] = prod;"),
    ("awl_sums_instead_of_multiplying", "prod *= alpha[(size_t)r * Bm1 + k];", "prod += alpha[(size_t)r * Bm1 + k];"),
    # acceptance probabilities, survivals, tau
    ("accept_prob_max", "a += P[v] < Q[v] ? P[v] : Q[v];", "a += P[v] > Q[v] ? P[v] : Q[v];"),
    ("tau_without_one", "double surv = 1.0, t = 1.0;", "double surv = 1.0, t = 0.0;"),
    ("survival_lags", "            surv *= a;\n            t += surv;", "            t += surv;\n            surv *= a;"),
    # branch construction
    ("anchor_may_be_drafted_token", "taken[yr[p]] = 1;", "taken[yr[p]] = 0;"),
    ("anchor_ties_to_highest", "if (bi < 0 || x > best) {", "if (bi < 0 || x >= best) {"),
    ("branch_parent_len_short", "row[4] = (k - 1) / F + 1;", "row[4] = (k - 1) / F;"),
    ("branch_head_len_short", "hl[k] = p + 1;", "hl[k] = p;"),
    # greedy verification
    ("greedy_ties_to_highest", "if (x > best) { /* strict", "if (x >= best) { /* strict"),
    ("greedy_compares_next_argmax", "while (a < B - 1 && y[(size_t)r * (B - 1) + a] == g[a])",
     "while (a < B - 1 && y[(size_t)r * (B - 1) + a] == g[a + 1])"),
    # branch match
    ("match_ignores_length", "if (head_len[(size_t)r * M + k] != n)", "if (head_len[(size_t)r * M + k] < n)"),
    ("match_last_duplicate", "for (int k = 0; k < M && hit < 0; ++k) {", "for (int k = 0; k < M; ++k) {"),
]


def _source():
    with open(SRC) as f:
        return f.read()


def _build_and_run(tmpdir, name, text):
    """Build one copy of the oracle and run the pins against it.
    Returns (pytest exit status, first failed pin or the output's tail)."""
    c = os.path.join(tmpdir, name + ".c")
    so = os.path.join(tmpdir, name + ".so")
    with open(c, "w") as f:
        f.write(text)
    subprocess.check_call(["gcc", *CFLAGS, c, "-o", so, "-lm"])
    env = dict(os.environ, D3D_ORACLE_LIB_OVERRIDE=so)
    res = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-m", "not gpu", "-p",
                          "no:cacheprovider", "-rf"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=900)
    failed = [ln.split()[1] for ln in res.stdout.splitlines() if ln.startswith("FAILED ")]
    return res.returncode, failed[0] if failed else res.stdout[-400:] + res.stderr[-400:]


def test_every_slip_is_planted_once():
    src = _source()
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name
        assert old != new, name


def test_every_planted_slip_fails_a_pin(tmp_path):
    src = _source()
    jobs = [("unchanged", src)] + [(name, src.replace(old, new)) for name, old, new in MUTANTS]
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        results = dict(zip([j[0] for j in jobs],
                           ex.map(lambda j: _build_and_run(str(tmp_path), *j), jobs)))
    rc, detail = results.pop("unchanged")
    assert rc == 0, "the unchanged copy must pass every pin: " + detail
    survived = [n for n, (rc, _) in results.items() if rc == 0]
    broken = ["%s (exit %d): %s" % (n, rc, d) for n, (rc, d) in results.items() if rc not in (0, 1)]
    assert not survived, "slips no pin catches: %s" % survived
    assert not broken, "children that did not end in failed pins: %s" % broken
