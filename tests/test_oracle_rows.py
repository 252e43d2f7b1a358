"""The row-split helper the full-size GPU parity tests use gives exactly the
oracle's own single-call results (same values, same row order)."""
import numpy as np
import pytest

import oracle_rows
import synthetic


@pytest.mark.parametrize("fmt,rows,cols,batch", [("q4k", 1000, 1024, 3), ("cb4", 777, 512, 2),
                                                 ("q4k", 5, 256, 1)])
def test_row_split_equals_one_call(orc, fmt, rows, cols, batch):
    W = (synthetic.q4k_weights(rows, cols, rows) if fmt == "q4k"
         else synthetic.cb4_weights(rows, cols, rows))
    kv = synthetic.cb4_table()
    xq = orc.quantize_q8(synthetic.activations(batch, cols, 3))
    one = (orc.matvec_q4k(W, xq, rows, cols, batch) if fmt == "q4k"
           else orc.matvec_cb4(W, kv, xq, rows, cols, batch))
    assert np.array_equal(oracle_rows.matvec(orc, fmt, W, kv, xq, rows, cols, batch), one)
    d1 = (orc.subdots_q4k(W, xq, rows, cols, batch) if fmt == "q4k"
          else orc.subdots_cb4(W, kv, xq, rows, cols, batch))
    assert np.array_equal(oracle_rows.subdots(orc, fmt, W, kv, xq, rows, cols, batch), d1)
