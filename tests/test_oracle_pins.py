"""The float64 oracle against what the pages and the mathematics fix (no GPU needed)."""
import pytest

from . import _pins

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.mark.parametrize("name", sorted(_pins.ALL_CHECKS))
def test_oracle_pin(oracle_lib, name):
    fails = _pins.ALL_CHECKS[name](oracle_lib)
    assert not fails, "\n".join(fails[:20])


@pytest.mark.skipif(not _pins.triton_philox_available(), reason="triton not importable")
def test_oracle_philox_matches_independent_implementation(oracle_lib):
    fails = _pins.check_philox_vs_triton(oracle_lib)
    assert not fails, "\n".join(fails[:20])
