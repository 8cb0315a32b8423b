"""The device's view of each mask must equal the oracle's visibility bit for
bit: attn_train_mask_pattern evaluates, through the same scheduling calls the
kernels make, which pairs the forward, the dK/dV pass and the dQ pass visit
unmasked -- in the form the kernels run for the problem (one-sided for full,
causal and TTT masks without key lengths) and in the general form -- TTT
suffix diagonals included.  Tile classes must be consistent: empty tiles hold
no visible pair, full tiles only visible pairs."""
import numpy as np
import pytest

import oracle
from attention_tcgen05_tmem_gb300 import binding
from tests.gpu_util import device

PLANES = ("forward", "dK/dV", "dQ", "forward (general)", "dK/dV (general)", "dQ (general)")

# causal, full, and the TTT mask at every step t = 0..6 of the EAGLE3 workload
CASES = ([("causal", 0, 128, 128), ("causal", 0, 1000, 1000), ("causal", 0, 300, 700),
          ("causal", 0, 700, 300), ("causal", 0, 257, 257), ("full", 0, 333, 129),
          ("full", 0, 1, 257)] +
         [("ttt", t, S, (t + 1) * S) for t, S in ((0, 260), (1, 300), (2, 5), (2, 384),
                                                  (3, 257), (4, 300), (4, 129), (5, 257),
                                                  (5, 640), (6, 640), (6, 200))])
# (mask, t, Sq, Skv, window, key length of the batch entry)
CASES_EXT = [("window", 0, 1000, 1000, (200, 0), None), ("window", 0, 900, 900, (130, 130), None),
             ("window", 0, 500, 777, (0, 300), None), ("window", 0, 450, 300, (5, 5), None),
             ("window", 0, 600, 600, (1, 0), 333), ("causal", 0, 700, 700, None, 321),
             ("full", 0, 333, 500, None, 129), ("causal", 0, 300, 300, None, 0),
             ("ttt", 2, 384, 1152, None, 200), ("ttt", 6, 260, 1820, None, 3),
             ("ttt", 4, 300, 1500, None, 129), ("ttt", 5, 257, 1542, None, 256)]


def _check(bits, tiles, want, kv_main):
    assert bits.shape[0] == len(PLANES)
    for p, name in enumerate(PLANES):
        if not np.array_equal(bits[p], want):
            q, kv = np.argwhere(bits[p] != want)[0]
            raise AssertionError(f"{name} schedule differs at q={q} kv={kv}")
    for qt in range(tiles.shape[0]):
        for kt in range(tiles.shape[1]):
            blk = want[qt * 128:(qt + 1) * 128, kt * 128:min((kt + 1) * 128, kv_main)]
            if tiles[qt, kt] == 0:
                assert blk.sum() == 0
            elif tiles[qt, kt] == 2:
                assert blk.all()


@pytest.mark.gpu
@pytest.mark.parametrize("mask,t,Sq,Skv,window,length", CASES_EXT)
def test_mask_pattern_window_and_lengths_bit_exact(mask, t, Sq, Skv, window, length):
    device()
    bits, tiles = binding.mask_pattern(Sq, Skv, mask, t, window=window, seq_length=length)
    want = oracle.mask(mask, t, Sq, Skv, window=window, length=length)
    _check(bits.cpu().numpy(), tiles.cpu().numpy(), want, Sq if mask == "ttt" else Skv)


@pytest.mark.gpu
@pytest.mark.parametrize("mask,t,Sq,Skv", CASES)
def test_mask_pattern_bit_exact(mask, t, Sq, Skv):
    device()
    bits, tiles = binding.mask_pattern(Sq, Skv, mask, t)
    want = oracle.mask(mask, t, Sq, Skv)
    _check(bits.cpu().numpy(), tiles.cpu().numpy(), want, Sq if mask == "ttt" else Skv)
