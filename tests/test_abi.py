"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
function include/markov.h declares; argument errors are reported without
touching a device."""
import ctypes

import pytest

from tests.conftest import has_gpu


@pytest.fixture(scope="module")
def L():
    from draft_token_markov_gb300 import api
    return api.lib()


def test_header_symbols_exported(L):
    from draft_token_markov_gb300 import api
    names = api.header_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(7):
        assert L.markov_status_string(code)
    assert L.markov_status_string(99) == b"unknown status"


def test_argument_errors_without_launch(L):
    assert L.markov_plan_set_path(None, 0) == 1
    assert L.markov_chain_max_rows(None) == -1
    assert L.markov_plan_query(None, 0) == -1
    assert L.markov_plan_status(None) == 1
    assert L.markov_device_math(9, None, None, 4, None) == 1
    assert L.markov_noise_fork(None, None, None, None, 1, None) == 1
    args = [None, None, 0, 0, None, None, None, None, None, None, 1, 0, 1.0, -1.0, None, 0,
            None, 0, 0, None]
    assert L.markov_chain_sample(*args) == 1


def test_plan_desc_validation(L):
    from draft_token_markov_gb300.api import _Desc
    h = ctypes.c_void_p()
    bad = [(4097, 256, 8, 8), (129280, 96, 8, 8), (129280, 256, 0, 8), (129280, 256, 17, 8),
           (129280, 256, 8, 0), (300000, 256, 8, 8)]
    for V, r, N, R in bad:
        d = _Desc(V, r, N, R, 0, 0)
        assert L.markov_plan_create(ctypes.byref(d), ctypes.byref(h)) == 1
        assert not h.value


@pytest.mark.skipif(has_gpu(), reason="checks the no-device answer")
def test_plan_create_without_device(L):
    from draft_token_markov_gb300.api import _Desc
    h = ctypes.c_void_p()
    d = _Desc(4096, 64, 4, 1, 0, 0)
    assert L.markov_plan_create(ctypes.byref(d), ctypes.byref(h)) == 6
