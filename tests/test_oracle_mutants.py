"""Plausible mistakes planted in the oracle (on the CPU) must fail a pin.

Each mutant is a one-line edit of a temporary copy of oracle/oracle.c: a
dropped scale, a wrong mask boundary, a wrong operand, a sign flip, a wrong
varlen offset. The copy is compiled and bound in place of the real oracle, and
the pin battery from test_oracle_pins.py is run against it; at least one pin
must fail. The real oracle must pass the same battery.
"""
import multiprocessing
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = [
    ("drop scale in scores", "return J->scale * dot(qi, kj, J->d);", "return dot(qi, kj, J->d);"),
    ("strict causal boundary", "if (J->wr >= 0 && j > i + delta + J->wr) return 0;",
     "if (J->wr >= 0 && j >= i + delta + J->wr) return 0;"),
    ("top-left causal alignment", "int delta = lk - lq;", "int delta = 0;"),
    ("window left bound off by one", "if (J->wl >= 0 && j < i + delta - J->wl) return 0;",
     "if (J->wl >= 0 && j <= i + delta - J->wl) return 0;"),
    ("window left bound on the wrong side", "if (J->wl >= 0 && j < i + delta - J->wl) return 0;",
     "if (J->wl >= 0 && j < i + delta + J->wl) return 0;"),
    ("causal ignored when a right window is given", "J->wr = causal ? 0 : wr;", "J->wr = wr >= 0 ? wr : (causal ? 0 : wr);"),
    ("LSE without the max", "return m + log(sum);", "return log(sum);"),
    ("base-2 exponential", "sum += exp(score(J, b, h, i, j) - m);", "sum += exp2(score(J, b, h, i, j) - m);"),
    ("O sums keys instead of values", "const double *vj = J->v + row_off_kv(J, b, j, kvh(J, h), J->Lk);\n        for (int c = 0; c < dv; c++) out[c]",
     "const double *vj = J->k + row_off_k(J, b, j, kvh(J, h), J->Lk);\n        for (int c = 0; c < dv; c++) out[c]"),
    ("score uses key row i", "const double *kj = J->k + row_off_k(J, b, j, kvh(J, h), J->Lk);\n    return",
     "const double *kj = J->k + row_off_k(J, b, i < J->Lk ? i : 0, kvh(J, h), J->Lk);\n    return"),
    ("keys of sequence b at its query offset", "if (J->cu) return ((long)(J->cuk[b] + j) * J->Hkv + hk) * J->d;",
     "if (J->cu) return ((long)(J->cu[b] + j) * J->Hkv + hk) * J->d;"),
    ("key length of sequence b from the query offsets",
     "static int seq_lk(const job_t *J, int b) { return J->cu ? J->cuk[b + 1] - J->cuk[b] : J->Lk; }",
     "static int seq_lk(const job_t *J, int b) { return J->cu ? J->cu[b + 1] - J->cu[b] : J->Lk; }"),
    ("block mask column from the query index", "if (!J->bmask[((long)hm * rows + i / J->bm_q) * cols + j / J->bm_k]) return 0;",
     "if (!J->bmask[((long)hm * rows + i / J->bm_q) * cols + i / J->bm_k]) return 0;"),
    ("block mask of head 0 for every head", "int hm = J->bm_h == 1 ? 0 : h;", "int hm = 0;"),
    ("interleaved head groups", "static int kvh(const job_t *J, int h) { return h / (J->H / J->Hkv); }",
     "static int kvh(const job_t *J, int h) { return h % J->Hkv; }"),
    ("dK/dV from the group's first query head only", "for (int hq = hk * g; hq < hk * g + g; hq++)",
     "for (int hq = hk * g; hq < hk * g + 1; hq++)"),
    ("dS sign flip", "return p * (dot(doi, vj, J->dvh) - J->D_all[st]);", "return p * (dot(doi, vj, J->dvh) + J->D_all[st]);"),
    ("D dropped", "J->D_all[st] = dot(", "J->D_all[st] = 0.0 * dot("),
    ("dQ without scale", "for (int c = 0; c < d; c++) dqi[c] *= J->scale;", ""),
    ("O written with the q/k head dim", "row_out(J, b, h, i, lse, J->o + row_off_v(J, b, i, h, J->Lq));",
     "row_out(J, b, h, i, lse, J->o + row_off(J, b, i, h, J->Lq));"),
    ("dK without scale", "for (int c = 0; c < d; c++) dkj[c] *= J->scale;", ""),
    ("dV weighted by dS", "dvj[c] += p * dor[c];", "dvj[c] += ds * dor[c];"),
    ("dK from dO instead of Q", "dkj[c] += ds * qr[c];", "dkj[c] += ds * dor[c];"),
    ("varlen row offset ignores start", "if (J->cu) return ((long)(J->cu[b] + i) * J->H + h) * J->d;",
     "if (J->cu) return ((long)(i) * J->H + h) * J->d;"),
    ("varlen LSE offset ignores start", "if (J->cu) return (long)h * J->cu[J->B] + J->cu[b] + i;",
     "if (J->cu) return (long)h * J->cu[J->B] + i;"),
]

BATTERY = [
    (pins.test_golden_hand_example, (False,)),
    (pins.test_golden_hand_example, (True,)),
    (pins.test_fwd_matches_textbook_softmax, (2, 3, 5, 5, 4, False)),
    (pins.test_fwd_matches_textbook_softmax, (1, 2, 7, 11, 8, True)),
    (pins.test_causal_first_row_returns_v0, ()),
    (pins.test_bottom_right_causal_with_more_queries, ()),
    (pins.test_varlen_is_per_sequence_attention, ()),
    (pins.test_bwd_finite_differences, (3, 4, False)),
    (pins.test_bwd_finite_differences, (7, 8, True)),
    (pins.test_bwd_finite_differences_rectangular_and_varlen, ()),
    (pins.test_bwd_column_sums, ()),
    (pins.test_fwd_matches_textbook_softmax_value_dim, (2, 3, 5, 5, 4, 3, False)),
    (pins.test_bwd_finite_differences_value_dim, (True,)),
    (pins.test_fwd_grouped_heads_match_textbook, (1, 6, 3, 7, 9, 3, True)),
    (pins.test_bwd_finite_differences_grouped_heads, (False,)),
    (pins.test_varlen_separate_key_lengths_is_per_sequence_attention, ()),
    (pins.test_window_matches_textbook_band, (9, 4, 3, 1)),
    (pins.test_window_matches_textbook_band, (7, 7, 2, 0)),
    (pins.test_zero_window_returns_the_diagonal_value, ()),
    (pins.test_bwd_finite_differences_window, (2, 1)),
    (pins.test_block_mask_matches_textbook, (True, 2, 3, True)),
    (pins.test_bwd_finite_differences_block_mask, (True,)),
    (pins.test_bwd_finite_differences_varlen_separate_keys, (True,)),
]


def run_battery():
    failed = []
    for fn, args in BATTERY:
        try:
            fn(*args)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError) as e:
            failed.append(f"{fn.__name__}{args}: {type(e).__name__}")
    return failed


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


def test_real_oracle_passes_battery():
    assert run_battery() == []


def _battery_in_child(so_path, conn):
    """Run the battery against the mutant library in a separate process: a
    mutant may write out of bounds (a wrong row stride), which must not corrupt
    the test process. Sends back the list of failed pins."""
    oracle._lib = oracle.bind(so_path)
    conn.send(run_battery())
    conn.close()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, src_text, tmp_path):
    assert src_text.count(old) == 1, f"mutation site for '{name}' not unique"
    mutated = src_text.replace(old, new)
    c_path = tmp_path / "mutant.c"
    c_path.write_text(mutated)
    so_path = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so_path),
                           str(c_path), "-lm", "-lpthread"])
    ctx = multiprocessing.get_context("spawn")
    parent, child = ctx.Pipe(duplex=False)
    proc = ctx.Process(target=_battery_in_child, args=(str(so_path), child))
    proc.start()
    child.close()
    try:
        failed = parent.recv() if parent.poll(300) else ["no result"]
    except EOFError:   # the child died before reporting: the mutant crashed a pin
        failed = ["child crashed"]
    proc.join(60)
    if proc.exitcode != 0:   # a crash of the mutant counts as a failed pin
        failed = failed + [f"child exit code {proc.exitcode}"]
    assert failed, f"mutant '{name}' passed every pin"
    shutil.rmtree(tmp_path, ignore_errors=True)
