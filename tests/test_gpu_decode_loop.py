"""Random-weight decode loop (the LM head's share of a decode step): a small
body, both sampling arms, the reported shares and the token feedback."""

import numpy as np
import pytest

from _helpers import to_device
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu

SMALL = dict(d=256, q=256, kv=64, ffn=512)


def test_decode_loop_reports_head_shares(fs, torch_cuda):
    torch = torch_cuda
    from lm_head_exact_gb300 import decode_loop
    fs.set_path(fs.FS_PATH_AUTO)
    W = to_device(synthetic.normal_blocks_bf16(1, 4096, 256, 0.02), torch)
    res = decode_loop.measure(W, batches=(1, 16), layers=2, steps=4, warmup=3, layer=SMALL)
    assert [r["B"] for r in res] == [1, 16]
    for r in res:
        for arm in ("fused", "unfused"):
            assert 0.0 < r[f"{arm}_head_us"] < r[f"{arm}_step_us"] * 1.5, r
            assert 0.0 < r[f"{arm}_head_share"] < 1.5, r
        assert np.isfinite(r["step_time_reduction"])


def test_decode_loop_feeds_sampled_ids_back(fs, torch_cuda):
    torch = torch_cuda
    from lm_head_exact_gb300 import decode_loop
    W = to_device(synthetic.normal_blocks_bf16(1, 4096, 256, 0.02), torch)
    loop = decode_loop.DecodeLoop(W, layers=2, layer=SMALL)
    ids0 = torch.arange(8, device="cuda", dtype=torch.int64) * 97
    temp = torch.ones(8, dtype=torch.float32, device="cuda")
    _, a = loop.run(ids0, temp, steps=3, fused=True, warmup=3)
    _, b = loop.run(ids0, temp, steps=3, fused=True, warmup=3)
    a, b = a.cpu().numpy(), b.cpu().numpy()
    np.testing.assert_array_equal(a, b)                 # deterministic given seed, step and inputs
    assert ((a >= 0) & (a < 4096)).all()
    # both arms draw the same Philox noise, so the unfused pipeline's
    # trajectory is the fused one's (away from near ties, which these seeded
    # inputs do not hit): the feedback loop carries the same tokens
    _, c = loop.run(ids0, temp, steps=3, fused=False, warmup=3)
    np.testing.assert_array_equal(c.cpu().numpy(), a)
