"""Pins of the oracle's greedy acceptance against what the page fixes.

"Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block",
section "Acceptance": a draft stands when the token chosen from the previous
row's logits equals it, and greedy verification gives, token for token, what
serial greedy decoding gives.  The checks below are hand-worked cases, numpy's
argmax (a library routine) on the one-row special case, and that serial-decoding
identity on a toy model; none re-types the oracle's loops.
"""
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_accept_cases():
    cases = []
    with open(os.path.join(GOLDEN, "accept_greedy.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, rows, drafts, expect = [part.strip() for part in line.split("|")]
            k, V = (int(t) for t in head.split())
            logits = np.array([[float(t) for t in row.split()] for row in rows.split(";")], np.float32)
            assert logits.shape == (k, V), line
            draft = [] if drafts == "-" else [int(t) for t in drafts.split()]
            a, nxt = (int(t) for t in expect.split())
            cases.append((logits, draft, a, nxt))
    return cases


@pytest.mark.parametrize("case", _golden_accept_cases())
def test_accept_matches_hand_worked_cases(case):
    logits, draft, a, nxt = case
    got_a, got_next, t = O.accept_greedy(logits, draft)
    assert (got_a, got_next) == (a, nxt)
    assert got_next == t[a - 1]


@pytest.mark.parametrize("seed", range(6))
def test_one_row_choice_is_numpy_argmax(seed):
    """k = 1: nothing to accept, a = 1, and the next token is the greedy
    choice, which under the tie readings is exactly numpy's argmax (lowest
    index among equal maxima, -0 == +0, the first NaN wins)."""
    rng = np.random.default_rng(seed)
    V = int(rng.integers(1, 3000))
    # few distinct values, so that ties are common
    row = rng.integers(-4, 5, V).astype(np.float32)
    if seed % 3 == 1:
        row[rng.integers(0, V, 3)] = np.float32(-0.0)
        row[rng.integers(0, V, 2)] = np.inf
    if seed % 3 == 2:
        row[rng.integers(0, V, 2)] = np.nan
    a, nxt, t = O.accept_greedy(row[None, :], [])
    assert a == 1
    assert nxt == t[0] == int(np.argmax(row))


def test_signed_zero_and_infinities():
    row = np.array([-np.inf, -0.0, 0.0, -1.0], np.float32)
    assert O.accept_greedy(row[None, :], [])[1] == 1 == int(np.argmax(row))
    row = np.array([3.0, np.inf, np.inf, np.nan, np.nan], np.float32)
    assert O.accept_greedy(row[None, :], [])[1] == 3 == int(np.argmax(row))


def _toy_model(rng, V):
    """A deterministic toy target: the logits after token u are table[u]."""
    return rng.standard_normal((V, V)).astype(np.float32)


@pytest.mark.parametrize("seed", range(12))
def test_accepted_tokens_equal_serial_greedy_decoding(seed):
    """Greedy mode gives what serial decoding gives, token for token: the
    accepted drafts followed by the next token are the first a tokens that
    serial greedy decoding emits after the pending token, and no longer prefix
    of the drafts would be."""
    rng = np.random.default_rng(100 + seed)
    V = int(rng.integers(2, 40))
    k = int(rng.integers(1, 17))
    table = _toy_model(rng, V)
    u = int(rng.integers(0, V))
    serial = []
    tok = u
    for _ in range(k):
        tok = int(np.argmax(table[tok]))
        serial.append(tok)
    # drafts: the serial continuation, corrupted from a random position on
    draft = list(serial[: k - 1])
    if k > 1 and seed % 4:
        j = int(rng.integers(0, k - 1))
        draft[j] = (draft[j] + 1 + int(rng.integers(0, V - 1))) % V
    rows = [u] + draft
    logits = np.stack([table[t] for t in rows])
    a, nxt, _ = O.accept_greedy(logits, draft)
    assert 1 <= a <= k
    emitted = draft[: a - 1] + [nxt]
    assert emitted == serial[:a]
    if a < k:
        assert draft[a - 1] != serial[a - 1]


def test_rejects_bad_sizes():
    with pytest.raises(ValueError):
        O.accept_greedy(np.zeros((3, 4), np.float32), [0])
