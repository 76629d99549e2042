"""The fp64 oracle pinned to facts outside itself (CPU only).

See tests/oracle_checks.py for what each check compares against."""
import pytest

import oracle_checks as oc  # noqa: E402


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check()


@pytest.mark.parametrize("V,K,T,seed,mask", [
    (2, 1, 1.0, 3, False), (4, 2, 0.5, 4, False), (6, 3, 1.7, 5, True), (5, 1, 0.05, 6, False)])
def test_exact_dense_grid(V, K, T, seed, mask):
    oc.check_exact_dense(V=V, K=K, T=T, seed=seed, mask=mask)


@pytest.mark.parametrize("V,K,T,seed", [(3, 1, 1.0, 8), (6, 3, 0.6, 9)])
def test_exact_onehot_grid(V, K, T, seed):
    oc.check_exact_onehot(V=V, K=K, T=T, seed=seed)


def test_chi_square_1e6():
    oc.check_chi_square()
