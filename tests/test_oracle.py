"""The FP64 oracle against its pins (CPU only)."""
import os

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load_library()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


MUTATIONS = {
    1: "exclusive causal bound",
    2: "interleaved query-head to kv-head map",
    3: "NHD / HND swapped",
    4: "sm_scale dropped",
    5: "wrong E4M3 exponent bias",
    6: "append positions shifted by one",
    7: "E4M3 encoding ties away from zero",
    8: "sink left out of the softmax denominator",
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m])
def test_planted_mistake_fails_a_pin(mutation, tmp_path):
    """Each planted mistake in a copy of the oracle fails at least one pin."""
    path = oracle.build(str(tmp_path / f"liboracle_m{mutation}.so"), mutation=mutation)
    mlib = oracle.load_library(path)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mlib)
        except (AssertionError, oracle.OracleError):
            failed.append(pin.__name__)
    assert failed, f"mutation '{MUTATIONS[mutation]}' passed every pin"


def test_rejects_bad_metadata(lib):
    d = pins.Dense(1, seq_lens=[5], q_lens=[1], Hq=2, Hkv=1, D=4, P=2)
    d.q_lens = np.array([6], np.int32)  # q_len > seq_len
    q_indptr = np.array([0, 6], np.int32)
    q = np.zeros((6, 2, 4), np.uint16)
    with pytest.raises(oracle.OracleError, match="q_len"):
        oracle.paged_decode(q, d.k_pool, d.v_pool, d.table, d.seq_lens, q_indptr, num_q_heads=2,
                            num_kv_heads=1, head_dim_qk=4, head_dim_v=4, page_size=2,
                            layout=oracle.NHD, sm_scale=1.0, lib=lib)
    bad = d.table.copy()
    bad[0, 1] = d.k_pool.shape[0] + 3
    with pytest.raises(oracle.OracleError, match="page"):
        oracle.paged_decode(d.q, d.k_pool, d.v_pool, bad, d.seq_lens, d.q_indptr, num_q_heads=2,
                            num_kv_heads=1, head_dim_qk=4, head_dim_v=4, page_size=2,
                            layout=oracle.NHD, sm_scale=1.0, lib=lib)


def test_empty_and_zero_length(lib):
    """A request with seq_len 0 and no query rows is a no-op; an empty batch
    returns empty arrays."""
    d = pins.Dense(2, seq_lens=[4, 3], q_lens=[1, 1], Hq=2, Hkv=1, D=4, P=2)
    out, lse = oracle.paged_decode(d.q[:0], d.k_pool, d.v_pool, d.table[:0], d.seq_lens[:0],
                                   np.zeros(1, np.int32), num_q_heads=2, num_kv_heads=1,
                                   head_dim_qk=4, head_dim_v=4, page_size=2, layout=oracle.NHD,
                                   sm_scale=1.0, lib=lib)
    assert out.shape == (0, 2, 4) and lse.shape == (0, 2)
    seq = np.array([4, 0], np.int32)
    qi = np.array([0, 1, 1], np.int32)
    out, lse = oracle.paged_decode(d.q[:1], d.k_pool, d.v_pool, d.table, seq, qi, num_q_heads=2,
                                   num_kv_heads=1, head_dim_qk=4, head_dim_v=4, page_size=2,
                                   layout=oracle.NHD, sm_scale=1.0, lib=lib)
    assert out.shape == (1, 2, 4) and np.isfinite(out).all()


def test_append_rejects_bad_metadata(lib):
    """q_len > seq_len writes nothing for that request; an out-of-range page
    id skips its rows; both report an error and leave other rows written."""
    P, Hkv, D = 4, 1, 4
    table = np.array([[0, 1], [2, 3]], np.int32)
    pool = np.zeros((4, P, Hkv, D), np.uint16)
    new = np.full((3, Hkv, D), 0x3F80, np.uint16)  # bf16 1.0
    kp, _, st = oracle.paged_append(new, None, table, np.array([1, 6], np.int32), np.array([0, 2, 3], np.int32),
                                    pool, num_kv_heads=Hkv, head_dim=D, page_size=P, layout=oracle.NHD, lib=lib)
    assert st == 2 and not kp[0:2].any() and (kp[3, 1] == 0x3F80).all()
    bad = table.copy()
    bad[1, 1] = 9
    kp, _, st = oracle.paged_append(new[:2], None, bad, np.array([1, 6], np.int32), np.array([0, 1, 2], np.int32),
                                    pool, num_kv_heads=Hkv, head_dim=D, page_size=P, layout=oracle.NHD, lib=lib)
    assert st == 3 and (kp[0, 0] == 0x3F80).all() and kp.sum() == 0x3F80 * D
