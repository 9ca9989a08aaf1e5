"""The FMA-pipe exponential of the forward kernels (ex2_fma), run on the GPU through the C ABI
self-test, against 2^x in float64 (numpy) and against the MUFU unit's ex2.approx."""
import numpy as np
import pytest
import torch

import exact_io_aware_gb300 as ea

pytestmark = pytest.mark.gpu


def test_fma_exponential_within_its_bound():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-125.0, 8.0, 1 << 20), np.arange(-125, 9, dtype=np.float64),
                        np.arange(-125, 9) + 0.5, [0.0, -0.0, 1e-30, -1e-30, 127.49]]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    y_fma, y_mufu = ea.attn_selftest_exp2(xd)
    assert ea.attn_device_status() == ea.ATTN_OK
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(y_fma.cpu().numpy().astype(np.float64) / want - 1.0)
    assert rel.max() < 7.5e-5 + 4e-7, rel.max()
    rel_m = np.abs(y_fma.cpu().numpy().astype(np.float64) / y_mufu.cpu().numpy().astype(np.float64) - 1.0)
    assert rel_m.max() < 1e-4


def test_fma_exponential_flushes_like_ex2_ftz():
    x = torch.tensor([-127.0, -130.0, -1e30, float("-inf")], device="cuda")
    y_fma, y_mufu = ea.attn_selftest_exp2(x)
    assert torch.equal(y_fma, torch.zeros_like(x))
    assert torch.equal(y_mufu, torch.zeros_like(x))
    empty = torch.empty(0, device="cuda")
    assert [t.numel() for t in ea.attn_selftest_exp2(empty)] == [0, 0]
