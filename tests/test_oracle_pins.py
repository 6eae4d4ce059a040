"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

from oracle import oracle as orc
from tests import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return orc.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_rejects_q_len_above_context(lib):
    q = np.zeros((3, 1, 4), np.float32)
    kc = np.zeros((1, 4, 1, 4), np.float32)
    with pytest.raises(orc.OracleError):
        orc.paged_attention(q, kc, kc, np.array([[0]], np.int32), np.array([2], np.int32),
                            np.array([0, 3], np.int32), 1, 1, 4, 4, 1.0, lib=lib)


def test_rejects_block_id_outside_pool(lib):
    q = np.zeros((1, 1, 4), np.float32)
    kc = np.zeros((1, 4, 1, 4), np.float32)
    with pytest.raises(orc.OracleError):
        orc.paged_attention(q, kc, kc, np.array([[5]], np.int32), np.array([2], np.int32),
                            np.array([0, 1], np.int32), 1, 1, 4, 4, 1.0, lib=lib)


def test_gather_rows_inverts_scatter(lib):
    rng = np.random.default_rng(0)
    dense = [rng.standard_normal((c, 2, 8)).astype(np.float32) for c in (5, 17, 1)]
    kc, _, table = oracle_pins.scatter_pages(dense, dense, 4, 7)
    got = orc.gather_rows(kc, table, np.array([5, 17, 1], np.int32), 4, 17)
    for s, d in enumerate(dense):
        np.testing.assert_array_equal(got[s, :d.shape[0]], d.reshape(d.shape[0], -1))
