"""The random-row gather probe (a measurement aid, no counterpart in the pages):
its per-row XOR equals numpy's on random bits, for every row size it takes,
with ids out of range clamped, and with more ids than one staging block."""
import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("row_bytes", [16, 32, 64, 128, 256, 512])
@pytest.mark.parametrize("n_ids", [1, 1000, 200003])
def test_probe_gather_xor(row_bytes, n_ids):
    rng = np.random.default_rng(row_bytes * 7 + n_ids)
    rows = 5000
    table = rng.integers(0, 2**32, size=rows * row_bytes // 4, dtype=np.uint64).astype(np.uint32)
    ids = rng.integers(-3, rows + 3, size=n_ids).astype(np.int32)  # a few out of range
    out = df2.probe_gather(torch.from_numpy(table.view(np.int32)).cuda(), row_bytes,
                           torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    t = table.reshape(rows, row_bytes // 4)
    want = np.bitwise_xor.reduce(t[np.clip(ids, 0, rows - 1)], axis=1)
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), want)
