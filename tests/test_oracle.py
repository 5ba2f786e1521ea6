"""The fp64 oracle against its pins (closed forms, torch SDPA, invariants)."""

import numpy as np
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_out_of_range_slot(orc):
    kc = np.zeros((1, 256, 1, 8), np.uint16)
    k = np.ones((1, 1, 8), np.uint16)
    with pytest.raises(oracle.OracleError):
        orc.kv_cache_write(k, k, np.array([256], np.int32), kc, kc.copy())
    with pytest.raises(oracle.OracleError):
        orc.kv_cache_write(k, k, np.array([-2], np.int32), kc, kc.copy())


def test_rejects_bad_table(orc):
    kc = np.zeros((2, 256, 1, 8), np.uint16)
    q = np.zeros((1, 1, 8), np.uint16)
    with pytest.raises(oracle.OracleError):
        orc.paged_attn_decode(q, kc, kc, np.array([300], np.int32), np.array([[0, 2]], np.int32), 1.0)
    with pytest.raises(oracle.OracleError):  # L > blocks in the table row
        orc.paged_attn_decode(q, kc, kc, np.array([600], np.int32), np.array([[0, 1]], np.int32), 1.0)


def test_rejects_negative_cached(orc):
    kc = np.zeros((2, 256, 1, 8), np.uint16)
    q = np.zeros((5, 1, 8), np.uint16)
    with pytest.raises(oracle.OracleError):  # n = 5 > L = 3
        orc.paged_attn_prefill(q, kc, kc, np.array([0, 5], np.int32), np.array([0, 3], np.int32),
                               np.array([[0]], np.int32), 1.0)


def test_row_sampling_matches_full(orc):
    import workloads
    w = workloads.make_prefill("t", 7, [300, 40], [100, 0], 4, 2, num_blocks=6, head_dim=16)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    orc.kv_cache_write(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    full = orc.paged_attn_prefill(w.q, kc, vc, w.cu_seqlens_q, w.cu_seqlens_k, w.block_tables, w.scale)
    rows = np.array([0, 5, 199, 200, 239])
    part = orc.paged_attn_prefill(w.q, kc, vc, w.cu_seqlens_q, w.cu_seqlens_k, w.block_tables, w.scale,
                                  rows=rows)
    assert np.array_equal(part[rows], full[rows])
    other = np.setdiff1d(np.arange(w.total_q), rows)
    assert np.isnan(part[other]).all()
