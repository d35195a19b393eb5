"""The benchmark's algorithmic FLOP and byte counts (the roofline numerators), checked on the CPU.

The closed forms in bench.py are pinned two ways: the per-chunk figures for d = 128, C = 64 that
the roofline quotes, and an independent brute-force count of the multiply-adds of every product
of the chunkwise form (Eq. 3-4 with the UT transform) under its causal mask, on small shapes.
"""
import itertools

import pytest

import bench


def _brute_force_macs(c, dk, dv):
    """Multiply-adds of one chunk of c tokens, product by product, counting only kept entries."""
    tril_incl = sum(1 for r, i in itertools.product(range(c), repeat=2) if i <= r)
    tril_strict = sum(1 for r, i in itertools.product(range(c), repeat=2) if i < r)
    intra = (tril_incl * dk      # A = Tril[(Q Gamma)(K / Gamma)^T], diagonal kept
             + tril_strict * dk  # L = StrictTril[diag(beta)(K Gamma)(K / Gamma)^T]
             + tril_incl * dk    # W = T diag(beta)(Gamma K): T lower triangular with its diagonal
             + tril_incl * dv)   # U = T diag(beta) V
    inter = (c * dk * dv         # W S
             + c * dk * dv       # (Gamma Q) S
             + c * dk * dv       # K~^T V~ (state update)
             + tril_incl * dv)   # A V~
    return intra, inter


@pytest.mark.parametrize("c,dk,dv", [(1, 2, 3), (3, 2, 2), (5, 4, 3), (16, 8, 8), (64, 128, 128)])
def test_prefill_flops_equal_brute_force_count(c, dk, dv):
    fl = bench.prefill_flops([c], 1, dk, dv, C=c)
    intra, inter = _brute_force_macs(c, dk, dv)
    inverse = c ** 3 / 3.0  # the triangular inverse, counted by convention
    assert fl["intra"] == pytest.approx(2 * intra + inverse, rel=1e-12)
    assert fl["inter"] == pytest.approx(2 * inter, rel=1e-12)


def test_prefill_flops_headline_figures():
    fl = bench.prefill_flops([64], 1, 128, 128)
    assert fl["intra"] == pytest.approx(2_200_917.33, abs=0.01)
    assert fl["inter"] == 6_823_936
    assert fl["total"] / 64 == pytest.approx(141_013.3, abs=0.1)  # per token-head
    # T = 4096, H = 32: 64 full chunks per head
    assert bench.prefill_flops([4096], 32, 128, 128)["total"] == pytest.approx(9_024_853.33 * 64 * 32, rel=1e-9)


def test_ragged_chunks_and_bytes():
    assert bench.chunk_lengths([5, 0, 64, 65, 130], 64) == [5, 64, 64, 1, 64, 64, 2]
    assert bench.chunk_lengths_count([5, 0, 64, 65, 130]) == [1, 0, 1, 2, 3]
    by = bench.prefill_bytes(T=4096, N=1, H=32, dk=128, dv=128, io_bytes=2, with_s0=False, with_sT=True)
    assert by["total"] == 4096 * 32 * 1282 + 32 * 128 * 128 * 4  # per token-head 1,282 B; S_T once
    assert bench.decode_bytes(256, 32, 128, 2) == 256 * 32 * 132_354
