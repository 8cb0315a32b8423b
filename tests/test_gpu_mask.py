"""The device's view of each mask (both the row-side schedule of the forward
and dQ passes and the column-side schedule of the dK/dV pass, TTT suffix
diagonals included) must equal the oracle's visibility bit for bit, and the
tile classes must be consistent: empty tiles hold no visible pair, full tiles
only visible pairs."""
import numpy as np
import pytest

import oracle
from attention_tcgen05_tmem_gb300 import binding
from tests.gpu_util import device

CASES = [("causal", 0, 128, 128), ("causal", 0, 1000, 1000), ("causal", 0, 300, 700),
         ("causal", 0, 700, 300), ("full", 0, 333, 129), ("ttt", 0, 260, 260),
         ("ttt", 1, 300, 600), ("ttt", 3, 257, 1028), ("ttt", 6, 640, 4480),
         ("ttt", 2, 5, 15)]
# (mask, t, Sq, Skv, window, key length of the batch entry)
CASES_EXT = [("window", 0, 1000, 1000, (200, 0), None), ("window", 0, 900, 900, (130, 130), None),
             ("window", 0, 500, 777, (0, 300), None), ("window", 0, 450, 300, (5, 5), None),
             ("window", 0, 600, 600, (1, 0), 333), ("causal", 0, 700, 700, None, 321),
             ("full", 0, 333, 500, None, 129), ("causal", 0, 300, 300, None, 0),
             ("ttt", 2, 384, 1152, None, 200), ("ttt", 6, 260, 1820, None, 3)]


def _check(bits, tiles, want, kv_main):
    np.testing.assert_array_equal(bits[0], want)
    np.testing.assert_array_equal(bits[1], want)
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
    bits = bits.cpu().numpy()
    want = oracle.mask(mask, t, Sq, Skv)
    np.testing.assert_array_equal(bits[0], want)
    np.testing.assert_array_equal(bits[1], want)
    tiles = tiles.cpu().numpy()
    kv_main = Sq if mask == "ttt" else Skv
    for qt in range(tiles.shape[0]):
        for kt in range(tiles.shape[1]):
            blk = want[qt * 128:(qt + 1) * 128, kt * 128:min((kt + 1) * 128, kv_main)]
            if tiles[qt, kt] == 0:
                assert blk.sum() == 0
            elif tiles[qt, kt] == 2:
                assert blk.all()
