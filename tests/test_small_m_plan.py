"""The few-token path's launch plan (host logic, no GPU): how the shared
dimension N is split over the CTAs of a cluster."""
from __future__ import annotations

import pytest


@pytest.fixture(scope="module")
def nb():
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300

    return backward_gemm_gb300


SHAPES = [(14336, 4096), (4096, 14336), (1536, 1536), (64, 64), (200, 320), (8960, 1536),
          (128, 8192), (65536, 128)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("sms,slots", [(152, 456), (152, 304), (152, 152), (8, 8)])
def test_every_rank_gets_work_and_all_of_n_is_covered(nb, N, K, sms, slots):
    S, per = nb.small_m_split(N, K, sms, slots)
    chunks = -(-N // 64)
    assert 1 <= S <= 16 and per >= 1
    assert S * per >= chunks          # the slices cover all of N
    assert (S - 1) * per < chunks     # the last rank's slice is not empty
    assert S <= chunks


@pytest.mark.parametrize("N,K,slots", [(14336, 4096, 456), (4096, 14336, 456),
                                       (14336, 4096, 304)])
def test_few_tiles_are_split_to_fill_the_gpu(nb, N, K, slots):
    """With fewer 256-column tiles than SMs, the split puts a CTA on most SMs
    (at least 70%), and all of them fit at once."""
    S, _ = nb.small_m_split(N, K, 152, slots)
    T = -(-K // 256)
    assert T * S >= 0.7 * 152
    assert T * S <= slots


@pytest.mark.parametrize("slots", [304, 456])
def test_long_n_prefers_fewer_longer_slices(nb, slots):
    """M = 16, N = 4096, K = 14336 (56 k-tiles of 64 stages): on GB300 clusters
    of 2 (one CTA per SM, 32 stages each) took 28.5 us, clusters of 5 (two CTAs
    on most SMs, 13 stages each) 31.0 us; the rule's fixed cost per CTA makes it
    take the former."""
    assert nb.small_m_split(4096, 14336, 152, slots) == (2, 32)


def test_one_stage_means_no_split(nb):
    assert nb.small_m_split(64, 4096, 152, 456) == (1, 1)


def test_rejects_bad_arguments(nb):
    import ctypes as C

    per = C.c_int(0)
    lib = nb.lib()
    assert lib.nf4_small_m_split(0, 64, 152, 456, C.byref(per)) == -1
    assert lib.nf4_small_m_split(64, 64, 0, 456, C.byref(per)) == -1
    assert lib.nf4_small_m_split(64, 64, 152, 456, None) == -1
