"""The Python binding refuses a table whose element type or shape does not
match its declared format before anything reaches the library: the kernels
index rows by the format's row bytes, so a uint8 code table passed as bf16
(or a short table) would be read past its end."""
import numpy as np
import pytest
import torch

import workloads as W
from hashed_gram_engram_gb300 import Engram


def _make(table, table_scale=None, rows=(5, 7), E=32):
    rows = np.asarray(rows, np.int64)
    D, H = 256, 2
    return Engram(dim=D, hc_mult=H, max_ngram_size=2, n_heads=len(rows), head_dim=E,
                  max_tokens=4, table=table, rows=rows, row_offset=W.row_offsets(rows),
                  wkv=torch.zeros((D * (H + 1), len(rows) * E), dtype=torch.bfloat16),
                  q_weight=torch.zeros((H, D), dtype=torch.bfloat16),
                  k_weight=torch.zeros((H, D), dtype=torch.bfloat16), device=0,
                  table_scale=table_scale, table_location=0)


@pytest.mark.parametrize("table,scale", [
    (torch.zeros((12, 32), dtype=torch.uint8), None),             # fp8 codes without scales
    (torch.zeros((12, 32), dtype=torch.bfloat16), torch.zeros((12, 1), dtype=torch.uint8)),
    (torch.zeros((11, 32), dtype=torch.bfloat16), None),          # fewer rows than the layout
    (torch.zeros((12, 16), dtype=torch.bfloat16), None),          # wrong head_dim
    (torch.zeros((32, 12), dtype=torch.bfloat16).t(), None),      # not contiguous
    (torch.zeros((12, 32), dtype=torch.uint8), torch.zeros((12, 2), dtype=torch.uint8)),
    (torch.zeros((12, 32), dtype=torch.uint8), torch.zeros((10, 1), dtype=torch.uint8)),
])
def test_mismatched_tables_are_refused(table, scale):
    with pytest.raises(ValueError):
        _make(table, scale)
