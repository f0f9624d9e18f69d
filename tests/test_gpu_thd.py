"""Padded packed rows <-> compact THD on the GPU vs the packing oracle, bit
for bit: bf16 rows of the query and key/value shapes, 16-byte int32 rows,
empty and full rows, lengths outside [0, S] (clamped), a single token."""
import numpy as np
import pytest
import torch

from oracle import thd
from block_sparse_gqa_msa_gb300 import api

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    ((3, 17, 64, 128), torch.bfloat16, [17, 0, 5]),
    ((8, 256, 4, 128), torch.bfloat16, [256, 200, 1, 0, 37, 255, 128, 3]),
    ((5, 33, 4), torch.int32, [-4, 40, 33, 0, 12]),
    ((1, 1, 8), torch.int32, [1]),
]


def _bits(t: torch.Tensor) -> np.ndarray:
    t = t.cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
    return t.numpy()


@pytest.mark.parametrize("shape,dtype,lens", CASES)
def test_pack_unpack_bit_exact(shape, dtype, lens):
    g = torch.Generator().manual_seed(hash(shape) & 0xFFFF)
    if dtype == torch.bfloat16:
        x = torch.randn(shape, generator=g).to(dtype)
    else:
        x = torch.randint(-1000, 1000, shape, generator=g, dtype=dtype)
    B, S = shape[0], shape[1]
    row_len = torch.tensor(lens, dtype=torch.int32)
    y, offs = api.pack_thd(x.to(DEV), row_len.to(DEV))
    torch.cuda.synchronize()
    ref_y = thd.pack_thd(_bits(x), lens)
    assert np.array_equal(_bits(y), ref_y)
    assert offs.cpu().numpy().tolist() == thd.row_offsets(lens, S).tolist()
    back = api.unpack_bshd(y, row_len.to(DEV), offs, S)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(back), thd.unpack_bshd(ref_y, lens, S))


def test_host_checks():
    x = torch.zeros(2, 4, 3, dtype=torch.int32, device=DEV)   # 12-byte rows
    with pytest.raises(api.MSAError):
        api.pack_thd(x, torch.tensor([1, 2], dtype=torch.int32, device=DEV))
