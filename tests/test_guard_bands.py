"""The guard bands the GPU parity tests put around every device array
(tests/_support.py), exercised on host memory: a write inside an array leaves
them intact, a write one element before or after it -- the kind of stray store
a ragged tail, a lone 4-bit nibble or a misaligned view could cause -- is
reported, with its offset."""

import numpy as np
import pytest
import torch

import _support as S


@pytest.fixture(autouse=True)
def _on_host(monkeypatch):
    monkeypatch.setattr(S, "DEVICE", "cpu")
    S.guards_reset()
    yield
    S.guards_reset()


@pytest.mark.parametrize("dtype,shift", [(torch.float32, 0), (torch.float32, 1), (torch.uint8, 3),
                                         (torch.int16, 1), (torch.bfloat16, 0)])
def test_in_bounds_writes_keep_the_bands(dtype, shift):
    t = S.guarded_empty(1001, dtype, shift)
    assert t.numel() == 1001 and t.is_contiguous()
    buf = S._GUARDED[-1][0]
    assert t.data_ptr() - buf.data_ptr() == S.GUARD + shift * t.element_size()
    t.zero_()
    t[-1] = 1
    S.assert_guards_intact()


@pytest.mark.parametrize("where", [-1, 0])
def test_a_store_beside_the_array_is_caught(where):
    a = S.dev(np.arange(37, dtype=np.float32), shift=1)
    S.zeros(5)
    buf, start, end = S._GUARDED[0]
    el = 4
    at = start - el if where < 0 else end      # the element just before / just after
    buf[at:at + el] = torch.tensor([1.0]).view(torch.uint8)
    with pytest.raises(AssertionError, match="array 0"):
        S.assert_guards_intact()
    assert a.numel() == 37


def test_dev_round_trips_values():
    x = np.random.default_rng(0).normal(size=(3, 5)).astype(np.float32)
    t = S.dev(x)
    assert np.array_equal(t.numpy(), x)
    s = S.scalar_i32(41)
    assert int(s.item()) == 41
    S.assert_guards_intact()
