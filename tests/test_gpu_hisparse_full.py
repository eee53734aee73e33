"""Mixed-residency decode (resolve + sparse MLA) at the benchmark's full context lengths.

Six requests of the HiSparse workload (contexts of 550K to 1.03M tokens, the last 4096 resident,
4096 hot slots each, top-2048 indices with 80 % step-to-step overlap, Zipf(1.1) over the older
tokens), three steps: every step's resolve is bit-exact against the oracle (rows, counters, the
whole LRU state, every pool byte), and the sparse MLA over the resolved rows matches the oracle
run on those rows."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_mla_gb300 import hs_check_flag, inputs
from dsa_sparse_mla_gb300.pipeline import DeviceHiSparse, pinned_uint8

from parity import check_mla

pytestmark = pytest.mark.gpu


def test_hisparse_full_context_lengths():
    steps = 3
    hw = inputs.config5(B=6, steps=steps, host_alloc=pinned_uint8)
    assert int(hw.seq_len.min()) > 500_000 and int(hw.seq_len.max()) > 1_000_000
    dh = DeviceHiSparse(hw)
    pool = hw.kv_pool.copy()
    stok = np.full((hw.B, hw.S), -1, np.int32)
    sstamp = np.full((hw.B, hw.S), -1, np.int32)
    t2s = np.full((hw.B, dh.ld_t2s), -1, np.int32)
    for step in range(steps):
        rows_ref, cnt_ref = oracle.hisparse_resolve(step, hw.idx[step], hw.seq_len, hw.resident_start,
                                                    hw.block_table, hw.host_rows, pool, hw.slot_row, stok,
                                                    sstamp, t2s)
        dh.step(step)
        torch.cuda.synchronize()
        assert hs_check_flag(dh.err) == 0, step
        assert np.array_equal(dh.rows.cpu().numpy(), rows_ref), step
        assert np.array_equal(dh.counters.cpu().numpy(), cnt_ref), step
        assert np.array_equal(dh.slot_token.cpu().numpy(), stok), step
        assert np.array_equal(dh.slot_stamp.cpu().numpy(), sstamp), step
        assert np.array_equal(dh.tok2slot.cpu().numpy(), t2s), step
        assert np.array_equal(dh.kv_pool.cpu().numpy(), pool), step
        if step == 0:
            assert (cnt_ref[:, 2] == hw.k).all()          # a cold buffer: every index misses
        else:
            assert (cnt_ref[:, 1] >= int(0.8 * hw.k)).all()  # the kept 80 % hit
        out_ref, lse_ref = oracle.sparse_mla(hw.q_mla[step], pool, rows_ref, hw.softmax_scale)
        check_mla(dh.out, dh.lse, out_ref, lse_ref)
