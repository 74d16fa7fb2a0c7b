"""The diagnostic fan-out copy the benchmark times as the ceiling of a one-read,
many-write stream: row r of the source lands in destination rows
floor(r*num/den) .. floor((r+1)*num/den) - 1, nothing else is written."""
import numpy as np
import pytest
import torch

import combine_ep_get_02_gb300 as ep

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("method", [0, 1])
@pytest.mark.parametrize("rows,row_bytes,num,den,sms", [
    (1000, 48, 17, 5, 0),        # ragged 16-byte chunks, fan-out 3.4
    (257, 14336, 7, 2, 0),       # dispatch-sized rows, fan-out 3.5
    (33, 4096, 1, 3, 5),         # fan-out below one: most rows are not written
    (9, 2064, 4, 1, 1),          # one SM
    (3000, 16384, 5, 4, 0),      # the widest rows the bulk method takes
])
def test_fanout_copy_places_rows(rows, row_bytes, num, den, sms, method):
    g = torch.Generator().manual_seed(rows)
    src = torch.randint(0, 256, (rows, row_bytes), dtype=torch.uint8, generator=g)
    n_dst = rows * num // den
    dst = torch.full((n_dst + 1, row_bytes), 0xA5, dtype=torch.uint8, device="cuda")
    ep.ep_diag_copy_fanout(src.cuda(), dst, rows, row_bytes, num, den, sms, method)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    exp = np.full((n_dst + 1, row_bytes), 0xA5, np.uint8)
    s = src.numpy()
    for r in range(rows):
        exp[r * num // den:(r + 1) * num // den] = s[r]
    assert np.array_equal(got, exp)


def test_fanout_copy_rejects_bad_arguments():
    src = torch.zeros(64, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for rows, rb, num, den in ((1, 24, 1, 1), (1, 16, 1, 0), (-1, 16, 1, 1), (1, 16, -1, 1)):
        with pytest.raises(ep.EpError):
            ep.ep_diag_copy_fanout(src, dst, rows, rb, num, den)
    with pytest.raises(ep.EpError):   # destination smaller than the fan-out needs
        ep.ep_diag_copy_fanout(src, dst, 4, 16, 5, 1)
