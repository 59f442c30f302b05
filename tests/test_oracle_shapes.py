"""The oracle over random small shapes, including the degenerate ones
(L = 1, N = 1, D = 1, batch = 1): the forward against brute-force unrolling
and the backward against torch.autograd (CPU only)."""
import numpy as np
import pytest
from hypothesis import given, settings
from hypothesis import strategies as st

import oracle
from tests import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@settings(max_examples=40, deadline=None)
@given(batch=st.integers(1, 3), L=st.integers(1, 12), D=st.integers(1, 5), N=st.integers(1, 9),
       seed=st.integers(0, 2**31 - 1))
def test_forward_against_unrolling(lib, batch, L, D, N, seed):
    pins.bruteforce_check(lib, np.random.default_rng(seed), batch, L, D, N)


@settings(max_examples=20, deadline=None)
@given(batch=st.integers(1, 2), L=st.integers(1, 8), D=st.integers(1, 4), N=st.integers(1, 7),
       seed=st.integers(0, 2**31 - 1))
def test_backward_against_autograd(lib, batch, L, D, N, seed):
    pins.bwd_against_autograd(lib, batch, L, D, N, seed)
