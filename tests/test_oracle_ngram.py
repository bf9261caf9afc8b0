"""Pins of the oracle's prompt-lookup (n-gram) drafting (CPU only).

The page's own example (a golden fixture, cited in the file) and hand-built histories
whose answers are fixed by the method as the page states it (take the last n tokens,
find them earlier in the history, propose what followed) and by the readings taken where
it is silent: the longest n first, the most recent occurrence, at most gamma tokens
clipped at the history's end.
"""
import torch

import oracle
from conftest import read_golden


def _draft(hist, max_n=3, min_n=1, gamma=4, Lmax=None, length=None):
    L = len(hist)
    Lmax = Lmax or L
    h = torch.full((1, Lmax), 0, dtype=torch.int32)
    h[0, :L] = torch.tensor(hist, dtype=torch.int32)
    d, n = oracle.ngram_draft(h, torch.tensor([L if length is None else length]), max_n, min_n,
                              gamma)
    return d[0].tolist(), int(n[0])


def test_page_example():
    rows = read_golden("ngram_prompt_lookup_example.txt")
    words, expected = rows[0], rows[1]
    vocab = {w: i for i, w in enumerate(dict.fromkeys(words + expected))}
    d, n = _draft([vocab[w] for w in words], max_n=3, min_n=1, gamma=3)
    assert n == 3
    assert d == [vocab[w] for w in expected]


def test_longest_ngram_wins_over_a_more_recent_shorter_match():
    # suffix (1, 2): the 2-gram occurs at 0 (followed by 7); the 1-gram 2 also occurs at
    # 5 (followed by 9), more recently, but the 2-gram is tried first
    d, n = _draft([1, 2, 7, 8, 4, 2, 9, 1, 2], max_n=2, min_n=1, gamma=2)
    assert (d, n) == ([7, 8], 2)
    # with 1-grams only, the most recent 2 (position 5) wins
    d, n = _draft([1, 2, 7, 8, 4, 2, 9, 1, 2], max_n=1, min_n=1, gamma=2)
    assert (d, n) == ([9, 1], 2)


def test_most_recent_occurrence_and_clipping_at_the_end():
    # suffix 5 occurs at 0 and 3; the most recent (3) is followed by 6, 5 and then the end
    d, n = _draft([5, 1, 2, 5, 6, 5], max_n=1, min_n=1, gamma=4)
    assert (d, n) == ([6, 5, -1, -1], 2)


def test_no_match_and_too_short_histories():
    assert _draft([1, 2, 3, 4], max_n=2, min_n=1, gamma=3) == ([-1, -1, -1], 0)
    assert _draft([7], max_n=1, min_n=1, gamma=2) == ([-1, -1], 0)
    assert _draft([], max_n=1, min_n=1, gamma=2, Lmax=4) == ([-1, -1], 0)
    # a match must leave a token after it: [3, 3] matches only at 0, followed by 3
    assert _draft([3, 3], max_n=1, min_n=1, gamma=2) == ([3, -1], 1)


def test_length_is_clamped_to_the_row():
    # a length past the row is read as the row's end; negative as empty
    assert _draft([4, 9, 4], max_n=1, min_n=1, gamma=2, length=10) == ([9, 4], 2)
    assert _draft([4, 9, 4], max_n=1, min_n=1, gamma=2, length=-3) == ([-1, -1], 0)
