"""The oracle, pinned to what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
import oracle_pins as P
from place_partial_rope_gb300 import synth


def test_worked_example():
    P.check_worked_example()


def test_formulations_agree_bitwise():
    P.check_formulations_agree()


@pytest.mark.parametrize("form", [oracle.GATHER_CHAIN, oracle.PAIR_ROTATION])
def test_complex_closed_form(form):
    P.check_complex_closed_form(form)


@pytest.mark.parametrize("form", [oracle.GATHER_CHAIN, oracle.PAIR_ROTATION])
def test_special_cases(form):
    P.check_special_cases(form)


@pytest.mark.parametrize("form", [oracle.GATHER_CHAIN, oracle.PAIR_ROTATION])
def test_invariants(form):
    P.check_invariants(form)


@pytest.mark.parametrize("form", [oracle.GATHER_CHAIN, oracle.PAIR_ROTATION])
def test_backward_is_transpose(form):
    P.check_backward_is_transpose(form)


@pytest.mark.parametrize("form", [oracle.GATHER_CHAIN, oracle.PAIR_ROTATION])
def test_adjoint_identity(form):
    P.check_adjoint_identity(form)


def test_oracle_rejects_bad_arguments():
    x, c, s, _ = synth.case((1, 2, 2, 8), 0, 8, "fp32", "BS1D", seed=1)
    with pytest.raises(ValueError):
        oracle.fwd(x, c, s, "fp32", 0, 10)        # end > D
    with pytest.raises(ValueError):
        oracle.fwd(x, c[..., :7], s[..., :7], "fp32", 0, 7)  # odd length
    with pytest.raises(ValueError):
        oracle.fwd(x, c[..., :4], s[..., :4], "fp32", 0, 8)  # r width != L
    bad = np.zeros((1, 3, 1, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.fwd(x, bad, bad, "fp32", 0, 8)    # S of r neither 1 nor S


def test_named_workload_tables_are_pair_duplicated_rotations():
    """The table recipe: cos/sin equal in lanes 2i and 2i+1, cos^2+sin^2 ~ 1,
    and the first pair's angle equals the position (theta = p / 10000^0)."""
    for name in ("tiny", "small_model"):
        wl = synth.WORKLOADS[name]
        _, c, s, _ = synth.workload_inputs(wl, with_grad=False)
        cf, sf = oracle.widen(c, wl.dtype), oracle.widen(s, wl.dtype)
        assert np.array_equal(cf[..., 0::2], cf[..., 1::2])
        assert np.array_equal(sf[..., 0::2], sf[..., 1::2])
        tol = 1e-6 if wl.dtype == "fp32" else 2e-2
        assert np.allclose(cf.astype(np.float64) ** 2 + sf.astype(np.float64) ** 2, 1.0, atol=tol)
        p = synth.positions(wl)
        assert np.allclose(cf[..., 0], np.cos(p.astype(np.float64)), atol=tol)
