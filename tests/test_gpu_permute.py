"""GPU parity of the dispatch (a2): the stable counting-sort scatter is
compared bit for bit with the oracle's stable sort (offsets, counts, the
padded row layout, perm, inv) and the copied rows with x."""
import numpy as np
import pytest
import torch

from mixture_experts_ffn_02_gb300 import synth
from mixture_experts_ffn_02_gb300.binding import Layer
from moe_check import padded_layout

pytestmark = pytest.mark.gpu

CASES = [
    # T, d, E, k, pad, skew
    (256, 64, 4, 2, 0, 0.0),
    (1000, 128, 4, 2, 0, 0.0),
    (4099, 512, 8, 2, 300, 0.0),      # ragged chunk, PAD tail
    (2000, 256, 64, 6, 0, 1.5),       # skewed: several experts empty or tiny
    (3000, 128, 128, 8, 0, 0.0),
    (1, 64, 4, 1, 0, 0.0),
    (130, 64, 256, 32, 5, 0.0),
    (777, 64, 16, 16, 0, 0.0),        # k = E
]


@pytest.mark.parametrize("T,d,E,k,pad,skew", CASES)
def test_permute_bit_exact(T, d, E, k, pad, skew):
    s = synth.MoEShape("perm", T=T, d=d, E=E, k=k, H=64, n_shared=0, H_shared=0)
    valid = None
    if pad:
        valid = torch.ones(T, dtype=torch.uint8)
        valid[T - pad:] = 0
    topk = synth.random_topk(T, E, k, seed=T, valid=valid, skew=skew)
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(1)).bfloat16()
    lay = Layer.create(s)
    lay.bufs.update(x=x.cuda(), topk_idx=topk.cuda())
    lay.bufs["x_perm"].fill_(7)       # pad rows must be overwritten with zeros
    lay.permute()
    torch.cuda.synchronize()
    assert lay.status() == 0
    offsets, row_offsets, row_of_pair, perm_padded = padded_layout(topk.numpy(), E)
    b = lay.bufs
    np.testing.assert_array_equal(b["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(b["counts"].cpu().numpy(), np.diff(offsets))
    np.testing.assert_array_equal(b["row_offsets"].cpu().numpy(), row_offsets)
    R = int(row_offsets[-1])
    assert R <= lay.R_cap
    np.testing.assert_array_equal(b["inv"].cpu().numpy(), row_of_pair)
    np.testing.assert_array_equal(b["perm"][:R].cpu().numpy(), perm_padded)
    xp = b["x_perm"][:R].cpu()
    real_rows = perm_padded >= 0
    src_tok = perm_padded[real_rows] // k
    assert torch.equal(xp[torch.from_numpy(real_rows)], x[torch.from_numpy(src_tok)])
    assert (xp[torch.from_numpy(~real_rows)].float() == 0).all()


def test_permute_bad_index_sets_status():
    T, E, k = 64, 4, 2
    s = synth.MoEShape("perm", T=T, d=64, E=E, k=k, H=64, n_shared=0, H_shared=0)
    topk = synth.random_topk(T, E, k, seed=3)
    topk[10, 1] = 9
    lay = Layer.create(s)
    lay.bufs.update(x=torch.zeros(T, 64, dtype=torch.bfloat16, device="cuda"),
                    topk_idx=topk.cuda())
    lay.permute()
    assert lay.status() == 8          # MOE_ERR_INDEX
    assert int(lay.bufs["counts"].sum()) == T * k - 1
