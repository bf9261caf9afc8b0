"""Prompt-lookup (n-gram) drafting on the GPU against the oracle: the proposed tokens and
their counts are integers and must be identical."""
import pytest
import torch

import oracle
import speculative_decoding_verify_sv_gb300 as sv

pytestmark = pytest.mark.gpu


def _histories(B, Lmax, vocab, seed):
    g = torch.Generator().manual_seed(seed)
    hist = torch.randint(0, vocab, (B, Lmax), generator=g, dtype=torch.int32)
    lens = torch.randint(0, Lmax + 1, (B,), generator=g, dtype=torch.int32)
    lens[0], lens[1], lens[2] = 0, 1, Lmax
    # repeated segments, so that longer n-grams find matches: every other sequence ends
    # with a copy of an earlier window of random length
    for b in range(3, B, 2):
        L = int(lens[b])
        k = int(torch.randint(2, 8, (1,), generator=g))
        if L > 4 * k:
            s = int(torch.randint(0, L - 2 * k, (1,), generator=g))
            hist[b, L - k:L] = hist[b, s:s + k].clone()
    return hist, lens


@pytest.mark.parametrize("B,Lmax,vocab,max_n,min_n,gamma,seed", [
    (64, 300, 6, 3, 1, 4, 1),        # small vocabulary: matches for every n
    (32, 2048, 50, 4, 2, 5, 2),
    (256, 8192, 200, 3, 1, 4, 3),    # long histories, a batch as large as the ragged one
    (16, 512, 3, 32, 1, 63, 4),      # the largest n-gram and gamma
])
def test_ngram_matches_oracle(cuda_ok, B, Lmax, vocab, max_n, min_n, gamma, seed):
    hist, lens = _histories(B, Lmax, vocab, seed)
    sv.sv_read_device_status()
    d, n = sv.sv_ngram_draft(hist.cuda(), lens.cuda(), max_n, min_n, gamma)
    torch.cuda.synchronize()
    rd, rn = oracle.ngram_draft(hist, lens, max_n, min_n, gamma)
    assert torch.equal(n.cpu(), rn)
    assert torch.equal(d.cpu(), rd)
    assert int((rn > 0).sum()) > B // 4  # the cases do exercise matches
    assert sv.sv_read_device_status() == 0


def test_ngram_length_out_of_range_is_clamped_and_reported(cuda_ok):
    hist = torch.tensor([[4, 9, 4, 1, 1, 1, 1, 1], [2, 5, 2, 5, 2, 7, 7, 7]], dtype=torch.int32)
    lens = torch.tensor([-2, 20], dtype=torch.int32)
    sv.sv_read_device_status()
    d, n = sv.sv_ngram_draft(hist.cuda(), lens.cuda(), 2, 1, 3)
    torch.cuda.synchronize()
    rd, rn = oracle.ngram_draft(hist, lens, 2, 1, 3)
    assert torch.equal(d.cpu(), rd) and torch.equal(n.cpu(), rn)
    assert sv.sv_read_device_status() & sv.SV_DEV_BAD_PREFIX
