"""Pins of the oracle's LoRA dropout on the bypass input
("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 5 training config;
"第 09 期 | QLoRA 4-bit 量化微调" LoraConfig: lora_dropout = p).

  * the oracle's Philox4x64-10, written from the published definition, equals
    numpy's Philox bit generator (a library routine) output for output,
    including far counters;
  * the keep mask is the stated rule applied to numpy's stream, and its keep
    rate is 1 - p within statistical bounds; p = 0 keeps everything;
  * forward and backward with a fixed mask equal torch fp64 autograd of
    y = x W^T + ((x * keep) / (1 - p)) A^T B^T alpha/r;
  * with p = 0 the dropout path is the plain oracle exactly.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle as orc


@pytest.mark.parametrize("seed", [0, 1234, 2 ** 40 + 7, 2 ** 64 - 1])
def test_philox_stream_equals_numpy(seed):
    raw = np.random.Philox(key=seed).random_raw(64)
    assert [orc.philox_stream(seed, o) for o in range(64)] == [int(v) for v in raw]
    for o in (4096 + 1, 2 ** 33 + 2, 2 ** 40 + 3):
        far = np.random.Philox(key=seed, counter=o // 4).random_raw(4)
        assert orc.philox_stream(seed, o) == int(far[o % 4])


def _keep_from_numpy(seed, p, M, K):
    n = M * K
    raw = np.random.Philox(key=seed).random_raw((n + 1) // 2)
    u = np.empty(2 * raw.size, dtype=np.uint64)
    u[0::2] = raw & 0xFFFFFFFF
    u[1::2] = raw >> np.uint64(32)
    p32 = min(int(np.floor(p * 2.0 ** 32 + 0.5)), 2 ** 32 - 1)
    return (u[:n] >= p32).astype(np.uint8).reshape(M, K)


@pytest.mark.parametrize("p", [0.0, 0.05, 0.1, 0.5])
def test_keep_mask_rule_and_rate(p):
    M, K = 37, 320
    keep = orc.dropout_keep(77, p, M, K)
    assert np.array_equal(keep, _keep_from_numpy(77, p, M, K))
    big = orc.dropout_keep(5, p, 1024, 1024)
    rate = big.mean()
    sd = np.sqrt(p * (1 - p) / big.size)
    assert abs(rate - (1 - p)) <= 6 * sd + 1e-12
    if p == 0.0:
        assert big.all()


def _bf16(shape, std, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("M,K,N,r,p", [(5, 128, 64, 4, 0.1), (7, 64, 192, 8, 0.3),
                                       (3, 256, 128, 16, 0.05)])
def test_dropout_forward_backward_match_torch_autograd(M, K, N, r, p):
    x, w, A = _bf16((M, K), 1.0, 1), _bf16((N, K), 0.02, 2), _bf16((r, K), 0.01, 3)
    B, dY = _bf16((N, r), 0.01, 4), _bf16((M, N), 1.0, 5)
    alpha = 2.0 * r
    keep = orc.dropout_keep(9, p, M, K)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    At = torch.tensor(A, dtype=torch.float64, requires_grad=True)
    Bt = torch.tensor(B, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(keep, dtype=torch.float64)
    xd = xt * kt / (1.0 - p)
    y = F.linear(xt, torch.tensor(w, dtype=torch.float64)) + F.linear(F.linear(xd, At), Bt) * (
        alpha / r)
    y.backward(torch.tensor(dY, dtype=torch.float64))
    y_o, t_o = orc.linear_fwd(x, w, A, B, alpha, keep=keep, p=p)
    np.testing.assert_allclose(y_o, y.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(t_o, (xd.detach() @ At.detach().T).numpy(), rtol=1e-12,
                               atol=1e-12)
    ref = orc.linear_bwd(x, dY, w, A, B, alpha, keep=keep, p=p)
    for name, got in (("dX", xt.grad), ("dA", At.grad), ("dB", Bt.grad)):
        np.testing.assert_allclose(ref[name], got.numpy(), rtol=1e-11, atol=1e-11,
                                   err_msg=name)


def test_zero_probability_is_the_plain_layer():
    M, K, N, r = 6, 128, 64, 8
    x, w, A = _bf16((M, K), 1.0, 11), _bf16((N, K), 0.02, 12), _bf16((r, K), 0.01, 13)
    B, dY = _bf16((N, r), 0.01, 14), _bf16((M, N), 1.0, 15)
    keep = orc.dropout_keep(3, 0.0, M, K)
    a = orc.linear_bwd(x, dY, w, A, B, 16.0, keep=keep, p=0.0)
    b = orc.linear_bwd(x, dY, w, A, B, 16.0)
    for k in ("dX", "dA", "dB", "t", "u"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(orc.linear_fwd(x, w, A, B, 16.0, keep=keep, p=0.0)[0],
                          orc.linear_fwd(x, w, A, B, 16.0)[0])
