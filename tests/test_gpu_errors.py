"""Device-side metadata errors in pkv_attention: each bad request is skipped
(its rows keep their sentinel), reported in the device error word with the
same bit the oracle reports, and the other requests are unaffected."""
import numpy as np
import pytest

import oracle
import paged_kv_attention_05_gb300 as pkv
from paged_kv_attention_05_gb300 import workloads as W

pytestmark = pytest.mark.gpu

from gpu_util import DeviceStep, assert_close  # noqa: E402

BITS = pkv.DEV_ERR_BITS


def _case(mutate, expect_bit, bad_req):
    step = W.build(W.custom([40, 0, 300, 7], [1, 20, 1, 9], 8, 2, seed=321, bt_width=None))
    kc, vc = step.key_cache.copy(), step.value_cache.copy()
    assert oracle.write(step.k, step.v, kc, vc, step.slot_mapping) == 0
    good, err = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                 step.block_table, step.num_reqs, step.scale)
    assert err == 0
    mutate(step)
    ref, oerr = oracle.attention(step.q, kc, vc, step.query_start_loc, step.seq_lens,
                                 step.block_table, step.num_reqs, step.scale)
    assert oerr & expect_bit
    ds = DeviceStep(step)
    ds.write()
    assert pkv.pkv_get_error() == 0
    ds.attention()
    bits = pkv.pkv_get_error()
    assert bits & BITS[{1: "SLOT_RANGE", 2: "QSL", 4: "SEQ_LEN", 8: "BT_WIDTH",
                        16: "BLOCK_ID"}[expect_bit]]
    got = ds.out_f64()
    qsl = step.query_start_loc
    for r in range(step.num_reqs):
        rows = slice(int(qsl[r]), int(qsl[r + 1]))
        if r == bad_req:
            if expect_bit != oracle.ERR_BLOCK_ID:   # a bad block id leaves rows unspecified
                assert np.isnan(got[rows]).all(), "rows of a skipped request were written"
        else:
            assert_close(got[rows], good[rows], "request %d" % r)


def test_seq_len_below_query_len():
    def m(step):
        step.seq_lens[1] = 5          # 20 query rows, seq_len 5
    _case(m, oracle.ERR_SEQ_LEN, 1)


def test_block_table_row_too_short():
    def m(step):
        step.seq_lens[0] = 16 * step.block_table.shape[1] + 1
    _case(m, oracle.ERR_BT_WIDTH, 0)


def test_block_id_outside_the_pool():
    def m(step):
        step.block_table[2, 3] = step.key_cache.shape[0] + 5
    _case(m, oracle.ERR_BLOCK_ID, 2)


def test_decreasing_query_start_loc():
    def m(step):
        step.query_start_loc[3] = step.query_start_loc[2] - 1   # request 2 has a negative length
    step = W.build(W.custom([40, 0, 300, 7], [1, 20, 1, 9], 8, 2, seed=321))
    ds = DeviceStep(step)
    ds.write()
    m(step)
    ds = DeviceStep(step)
    ds.attention()
    assert pkv.pkv_get_error() & BITS["QSL"]
