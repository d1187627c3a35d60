"""The canary helper on host tensors: writes inside a tensor leave the pads
intact, a write one element past either end is seen."""
import torch

from tests.canary import Canaries


def test_canaries_see_writes_outside_only():
    c = Canaries("cpu")
    a = c.tensor((3, 5), torch.bfloat16)
    b = c.tensor((7,), torch.float32)
    a.fill_(1.0)
    b.copy_(torch.arange(7.0))
    assert c.broken() == []
    assert a.data_ptr() % 16 == 0 and b.data_ptr() % 16 == 0     # the library's alignment rule
    raw, _ = c.bufs[1]
    raw.view(torch.float32)[1024 + 7] = 2.0       # the float right after b
    assert c.broken() == [1]
    c2 = Canaries("cpu")
    d = c2.tensor((4,), torch.float16)
    raw2, _ = c2.bufs[0]
    raw2[4095] = 0
    assert c2.broken() == [0] and d.numel() == 4
