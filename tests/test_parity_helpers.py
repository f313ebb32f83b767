"""CPU checks of the comparison helpers the GPU parity tests rely on: the
piecewise whole-tensor accumulator must give exactly what the direct
whole-array formulas give, whatever the pieces, and its worst-head value
must be the per-head relative error."""
import numpy as np
import torch

from tests.parity import WholeTensorError, device_compare, max_over_rms, rel_l2


def _data(seed=0, shape=(37, 5, 16)):
    g = torch.Generator().manual_seed(seed)
    ref = (torch.randn(shape, generator=g, dtype=torch.float64) * 3).float()
    x = (ref + 1e-3 * torch.randn(shape, generator=g, dtype=torch.float64)).to(torch.bfloat16)
    return x, ref


def test_pieces_add_up_to_the_whole_tensor():
    x, ref = _data()
    acc = WholeTensorError(5, torch.bfloat16)
    # uneven pieces along the token axis, and one piece split by heads
    acc.add(x[:10], ref[:10], head_axis=1)
    acc.add(x[10:30, :2], ref[10:30, :2], head_axis=1, heads=[0, 1])
    acc.add(x[10:30, 2:], ref[10:30, 2:], head_axis=1, heads=[2, 3, 4])
    acc.add(x[30:], ref[30:], head_axis=1)
    assert abs(acc.rel_l2() - rel_l2(x, ref)) <= 1e-12 * rel_l2(x, ref)
    assert abs(acc.max_over_rms() - max_over_rms(x, ref, torch.bfloat16)) <= 1e-12
    per = [rel_l2(x[:, h], ref[:, h]) for h in range(5)]
    h, w = acc.worst_head()
    assert h == int(np.argmax(per)) and abs(w - max(per)) <= 1e-12


def test_a_bad_head_is_found_and_fails_the_check():
    x, ref = _data(1)
    x = x.clone()
    x[:, 3] += 0.5  # one head far off
    acc = WholeTensorError(5, torch.bfloat16)
    acc.add(x, ref, head_axis=1)
    assert acc.worst_head()[0] == 3
    try:
        acc.check(torch.bfloat16, "planted")
    except AssertionError:
        return
    raise AssertionError("a head off by 0.5 passed the bf16 bounds")


def test_device_compare_equals_host_formulas():
    x, ref = _data(2)
    rel, mx = device_compare(x, ref)
    assert abs(rel - rel_l2(x, ref)) <= 1e-12
    assert abs(mx - max_over_rms(x, ref, torch.bfloat16)) <= 1e-12
    y = ref.to(torch.bfloat16)
    rel2, mx2 = device_compare(x, y, both_stored=True)
    assert abs(rel2 - rel_l2(x, y)) <= 1e-12
    assert abs(mx2 - max_over_rms(x, y, torch.bfloat16, 2)) <= 1e-12
