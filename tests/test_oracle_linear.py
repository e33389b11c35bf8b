"""Pins for the oracle's QLoRA linear forward and backward.

Pins used:
  * library special case: torch CPU float64 F.linear and autograd of the
    page formula y = x W^T + (x A^T) B^T alpha/r ("QLoRA and 4bit
    Quantization | QLoRA 与 4-bit 量化", Step 3) cross-check the oracle's
    hand-derived forward and backward;
  * the page fixture and its output/branch/gradient contracts (same page,
    Step 4 tests: test_lora_branch_contract, test_frozen_base_gradient_contract,
    test_qlora_output_contract);
  * special cases: B = 0 gives exactly the base output and dA == 0;
  * row independence (sampled rows equal the full result).
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).float().numpy()


def _case(M, K, N, r, seed=0, zero_b=False):
    x = _bf16((M, K), 1.0, seed + 1)
    w = _bf16((N, K), 0.02, seed + 2)
    A = _bf16((r, K), 0.01, seed + 3)
    B = np.zeros((N, r), np.float32) if zero_b else _bf16((N, r), 0.01, seed + 4)
    dY = _bf16((M, N), 1.0, seed + 5)
    return x, w, A, B, dY


def _torch_ref(x, w, A, B, dY, alpha):
    r = A.shape[0]
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64)
    At = torch.tensor(A, dtype=torch.float64, requires_grad=True)
    Bt = torch.tensor(B, dtype=torch.float64, requires_grad=True)
    y = F.linear(xt, wt) + F.linear(F.linear(xt, At), Bt) * (alpha / r)
    y.backward(torch.tensor(dY, dtype=torch.float64))
    return (y.detach().numpy(), xt.grad.numpy(), At.grad.numpy(), Bt.grad.numpy(),
            (xt.detach() @ At.detach().T).numpy())


@pytest.mark.parametrize("M,K,N,r", [(5, 128, 64, 4), (3, 64, 192, 8), (16, 256, 128, 16)])
def test_forward_matches_torch_fp64(M, K, N, r):
    x, w, A, B, dY = _case(M, K, N, r)
    y, t = orc.linear_fwd(x, w, A, B, alpha=2.0 * r)
    y_ref, _, _, _, t_ref = _torch_ref(x, w, A, B, dY, 2.0 * r)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(t, t_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("M,K,N,r", [(5, 128, 64, 4), (7, 64, 320, 16), (2, 192, 64, 2)])
def test_backward_matches_torch_autograd_fp64(M, K, N, r):
    x, w, A, B, dY = _case(M, K, N, r, seed=10)
    alpha = 16.0
    g = orc.linear_bwd(x, dY, w, A, B, alpha)
    _, dx_ref, da_ref, db_ref, t_ref = _torch_ref(x, w, A, B, dY, alpha)
    np.testing.assert_allclose(g["dX"], dx_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dA"], da_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dB"], db_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["t"], t_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["u"], dY.astype(np.float64) @ B.astype(np.float64),
                               rtol=1e-12, atol=1e-12)


def test_zero_b_gives_base_output_and_zero_dA():
    x, w, A, B, dY = _case(4, 128, 64, 8, zero_b=True)
    y, _ = orc.linear_fwd(x, w, A, B, alpha=16.0)
    base, _ = orc.linear_fwd(x, w, A, np.zeros_like(B), alpha=0.0)
    assert np.array_equal(y, base)
    np.testing.assert_allclose(y, x.astype(np.float64) @ w.astype(np.float64).T,
                               rtol=1e-12, atol=1e-12)
    g = orc.linear_bwd(x, dY, w, A, B, 16.0)
    assert np.all(g["dA"] == 0.0)
    assert np.any(g["dB"] != 0.0)


def test_lora_branch_changes_output():
    x, w, A, B, dY = _case(4, 128, 64, 8)
    y, _ = orc.linear_fwd(x, w, A, B, alpha=16.0)
    base, _ = orc.linear_fwd(x, w, A, np.zeros_like(B), alpha=16.0)
    assert y.shape == base.shape
    assert not np.allclose(y, base, atol=1e-6)


def test_sampled_rows_equal_full_result():
    x, w, A, B, dY = _case(9, 64, 128, 4)
    y, t = orc.linear_fwd(x, w, A, B, 8.0)
    rows = np.array([8, 0, 3], np.int64)
    ys, ts = orc.linear_fwd(x, w, A, B, 8.0, rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(ts, t[rows])
    g = orc.linear_bwd(x, dY, w, A, B, 8.0)
    gs = orc.linear_bwd(x, dY, w, A, B, 8.0, rows=rows)
    assert np.array_equal(gs["dX"], g["dX"][rows])
    assert np.array_equal(gs["dA"], g["dA"]) and np.array_equal(gs["dB"], g["dB"])


def test_p1_fixture_contracts(golden_dir):
    with open(os.path.join(golden_dir, "p1_fixture.json")) as f:
        fx = json.load(f)
    table = orc.codebook()
    idx = np.array(fx["indices"])
    w = (table[idx] * np.float32(fx["scale"])).astype(np.float32)
    A = np.array(fx["lora_A"], np.float32)
    B = np.array(fx["lora_B"], np.float32)
    x3 = np.array(fx["x"], np.float32)
    x = x3.reshape(-1, fx["in_features"])
    y, _ = orc.linear_fwd(x, w, A, B, fx["alpha"])
    out = y.reshape(*x3.shape[:-1], fx["out_features"])
    assert list(out.shape) == fx["expected_output_shape"]
    # explicit page formula evaluated by torch in float32 (the page's own check)
    xt = torch.tensor(x3)
    ref = F.linear(xt, torch.tensor(w)) + (xt @ torch.tensor(A).T) @ torch.tensor(B).T * (
        fx["alpha"] / fx["r"])
    np.testing.assert_allclose(out, ref.numpy(), atol=fx["output_atol"], rtol=0)
    base = F.linear(xt, torch.tensor(w)).numpy()
    assert not np.allclose(out, base, atol=1e-6)
    # gradients reach x, A, B; the NF4 state (indices, scale) is never written
    idx_before = idx.copy()
    dY = np.ones((x.shape[0], fx["out_features"]), np.float32)  # out.sum().backward()
    g = orc.linear_bwd(x, dY, w, A, B, fx["alpha"])
    assert np.any(g["dX"] != 0) and np.any(g["dA"] != 0) and np.any(g["dB"] != 0)
    assert np.array_equal(idx, idx_before)


def test_oracle_does_not_write_its_inputs():
    x, w, A, B, dY = _case(4, 64, 64, 4)
    copies = [a.copy() for a in (x, w, A, B, dY)]
    orc.linear_fwd(x, w, A, B, 8.0)
    orc.linear_bwd(x, dY, w, A, B, 8.0)
    for a, c in zip((x, w, A, B, dY), copies):
        assert np.array_equal(a, c)
    wq = _bf16((8, 128), 0.02, 1)
    q = orc.quantize_nf4(wq, group=256)
    before = (q.packed.copy(), q.absmax_code.copy(), q.scale2.copy())
    orc.dequant_bf16(q)
    assert all(np.array_equal(a, b) for a, b in zip(before, (q.packed, q.absmax_code, q.scale2)))
