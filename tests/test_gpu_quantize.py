"""GPU parity of quantisation and dequantisation against the CPU oracle.

Bit-exact: indices, packed bytes, int8 codes, second-level scales (or fp32
constants) and the dequantised bf16 weight."""
import numpy as np
import pytest
import torch

from bit_nf4_quantized_35_b300 import capi, inputs
from oracle import oracle

from .helpers import bf16_bits, unpack_nibbles

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    capi.load()


def _check_quant(W_cpu: torch.Tensor, group: int):
    """Quantise on the GPU and with the oracle; compare every output bit."""
    W = W_cpu.cuda().contiguous()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = capi.quantize_nf4(W, group=group, nonfinite_flag=flag)
    deq = capi.dequant(q)
    torch.cuda.synchronize()
    ref = oracle.quantize_nf4(W_cpu.float().numpy(), 64, group)
    assert np.array_equal(q.packed.cpu().numpy(), ref.packed), "packed bytes differ"
    if group > 0:
        assert np.array_equal(q.absmax_code.cpu().numpy(), ref.absmax_code), "codes differ"
        assert q.scale2.cpu().numpy().tobytes() == ref.scale2.tobytes(), "scale2 differs"
    else:
        assert q.absmax_f32.cpu().numpy().tobytes() == ref.absmax_f32.tobytes()
    assert np.array_equal(bf16_bits(deq).ravel(), oracle.dequant_bf16(ref).ravel()), \
        "dequantised bf16 differs"
    assert int(flag.item()) == (1 if ref.nonfinite else 0)
    return q, ref


def test_single_layer_fp32_weight():
    """256x256 fp32 weight N(0, 0.02), seed 0, block 64, group 256."""
    W = inputs.normal((256, 256), inputs.STD_W, inputs.SEED_W, torch.float32)
    _check_quant(W, 256)


@pytest.mark.parametrize("group", [0, 32, 64, 128, 256])
def test_groups_and_ragged_tail(group):
    # 37 rows x 192 cols = 111 blocks: one partial CTA, partial last group
    W = inputs.normal((37, 192), inputs.STD_W, 11, torch.bfloat16)
    _check_quant(W, group)


def test_edge_values():
    """Zero blocks, exact +-absmax, worked example 0.2, ties, denormals."""
    rows, cols = 8, 128
    W = torch.zeros(rows, cols, dtype=torch.float32)
    W[1, :64] = torch.linspace(-1, 1, 64)
    W[2, 0], W[2, 1], W[2, 2] = 0.5, -0.5, 0.1     # normalised 1, -1, 0.2
    cb = oracle.codebook()
    mids = (cb[:-1].astype(np.float64) + cb[1:]) / 2
    W[3, :15] = torch.tensor(mids, dtype=torch.float32)
    W[3, 15] = 1.0
    W[4, :64] = torch.full((64,), 1e-40)           # denormal block
    W[4, 3] = -3e-40
    W[5, 64:] = torch.randn(64) * 1e30
    W[6, :] = -0.0
    W[7, :64] = torch.tensor(np.nextafter(np.float32(mids), np.float32(2)).tolist()
                             + [1.0] * 49, dtype=torch.float32)
    q, ref = _check_quant(W, 256)
    idx = unpack_nibbles(ref.packed).reshape(rows, cols)
    assert idx[2, 0] == 15 and idx[2, 1] == 0 and idx[2, 2] == 9   # worked example
    assert np.all(idx[0] == 7)


def test_nonfinite_flag():
    W = inputs.normal((4, 128), inputs.STD_W, 5, torch.float32)
    W[1, 7] = float("nan")
    W[3, 70] = float("inf")
    Wc = W.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = capi.quantize_nf4(Wc, nonfinite_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 1
    ref = oracle.quantize_nf4(W.numpy(), 64, 256)
    assert ref.nonfinite == 2
    # blocks without non-finite entries are still bit-exact
    got = unpack_nibbles(q.packed.cpu().numpy()).reshape(4, 128)
    exp = unpack_nibbles(ref.packed).reshape(4, 128)
    for r, c0 in [(0, 0), (0, 64), (1, 64), (2, 0), (2, 64), (3, 0)]:
        assert np.array_equal(got[r, c0:c0 + 64], exp[r, c0:c0 + 64])


def test_bulk_matrix_with_outliers_full_size():
    """One full 4096x14336 bulk-quantisation matrix (0.1% +-10 sigma outliers)."""
    W = inputs.bulk_matrix(0)
    _check_quant(W, 256)


def test_projection_weight_full_size():
    W = inputs.normal((4096, 4096), inputs.STD_W, inputs.SEED_W, torch.bfloat16)
    _check_quant(W, 256)


def test_dequant_deterministic_and_buffers_const():
    W = inputs.normal((64, 256), inputs.STD_W, 3, torch.bfloat16).cuda()
    q = capi.quantize_nf4(W)
    before = [t.clone() for t in (q.packed, q.absmax_code, q.scale2)]
    a = capi.dequant(q)
    b = capi.dequant(q)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for x, y in zip(before, (q.packed, q.absmax_code, q.scale2)):
        assert torch.equal(x, y)


@pytest.mark.slow
def test_exhaustive_decision_rule_all_fp32_in_unit_interval():
    """Every fp32 x in [-1, 1] (about 2.13e9 values) quantised as the
    non-maximal element of a block whose absmax is exactly 1 (so w / a == x)
    gets the oracle's nearest-codepoint index."""
    per_block = 63
    chunk_blocks = 1 << 20
    ranges = [(0x00000000, 0x3F800000 + 1), (0x80000000, 0xBF800000 + 1)]
    for lo, hi in ranges:
        start = lo
        while start < hi:
            n = min(per_block * chunk_blocks, hi - start)
            nb = (n + per_block - 1) // per_block
            bits = torch.arange(start, start + nb * per_block, dtype=torch.int64, device="cuda")
            bits = torch.clamp(bits, max=hi - 1)
            vals = (bits.to(torch.int32)).view(torch.float32).view(nb, per_block)
            W = torch.cat([torch.ones(nb, 1, device="cuda"), vals], dim=1).contiguous()
            q = capi.quantize_nf4(W.view(nb, 64), group=0)
            p = q.packed.view(nb, 32)
            idx = torch.stack([p >> 4, p & 15], dim=2).view(nb, 64)[:, 1:].reshape(-1)[:n]
            ref = oracle.nearest_codes_bits(start, n)
            assert np.array_equal(idx.cpu().numpy(), ref), hex(start)
            start += n
