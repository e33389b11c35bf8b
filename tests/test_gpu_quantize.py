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


def _check_quant(W_cpu: torch.Tensor, group: int, block: int = 64, codebook: int = 0):
    """Quantise on the GPU and with the oracle; compare every output bit."""
    W = W_cpu.cuda().contiguous()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = capi.quantize_nf4(W, group=group, nonfinite_flag=flag, block=block, codebook=codebook)
    deq = capi.dequant(q)
    torch.cuda.synchronize()
    ref = oracle.quantize_nf4(W_cpu.float().numpy(), block, group, codebook=codebook)
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


@pytest.mark.parametrize("group", [0, 32, 64, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_block128_groups_and_ragged_tail(group, dtype):
    """128-weight blocks: 37 x 384 = 111 blocks (one partial CTA, a partial
    last group), bf16 and fp32 weights, every output bit."""
    W = inputs.normal((37, 384), inputs.STD_W, 12, dtype)
    W[5, 128:256] = 0.0  # an all-zero block
    _check_quant(W, group, block=128)


@pytest.mark.parametrize("fmt", [(64, 256), (64, 0), (128, 256)], ids=lambda f: f"b{f[0]}g{f[1]}")
def test_quantile_codebook_ragged(fmt):
    """The quantile-formula table (symmetric, no zero): 37 x 384 weights with
    an all-zero block and exact zeros inside blocks, every output bit."""
    W = inputs.normal((37, 384), inputs.STD_W, 13, torch.bfloat16)
    W[3, 128:256] = 0.0
    W[4, 5] = 0.0
    _check_quant(W, fmt[1], block=fmt[0], codebook=1)


def test_quantile_codebook_bulk_matrix_full_size():
    _check_quant(inputs.bulk_matrix(2), 256, codebook=1)


def test_block128_bulk_matrix_full_size():
    _check_quant(inputs.bulk_matrix(1), 256, block=128)


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


@pytest.mark.parametrize("a_bits", [0x3F80, 0x3C99, 0x0080, 0x44D5, 0x0003, 0x7F7F],
                         ids=["1", "0.0187", "min-normal", "1704", "subnormal", "max"])
@pytest.mark.parametrize("group", [256, 0])
def test_bf16_every_value_under_absmax(a_bits, group):
    """Every finite bf16 value w with |w| <= a, as the non-maximal elements of
    blocks of 64 whose absmax is a (the bf16 input path), bit-exact against
    the oracle on the same values."""
    pats = np.arange(0x10000, dtype=np.uint32)
    vals = (pats << 16).view(np.float32)
    a = np.array([a_bits << 16], dtype=np.uint32).view(np.float32)[0]
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= a)]
    n = -(-vals.size // 63) * 63
    vals = np.concatenate([vals, np.zeros(n - vals.size, np.float32)]).reshape(-1, 63)
    blocks = np.concatenate([np.full((vals.shape[0], 1), a, np.float32), vals], axis=1)
    W = torch.from_numpy(blocks.reshape(-1, 1024) if blocks.size % 1024 == 0 else blocks)
    _check_quant(W.to(torch.bfloat16), group)


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


def _f32_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float32).view(np.uint32)[0])


def _sweep(absmax: float, start: int, count: int, chunk_blocks: int = 1 << 20):
    """Quantise every binary32 weight with the `count` consecutive bit
    patterns from `start` as the non-maximal elements of blocks whose first
    element (the absmax) is `absmax`, and compare each index with the
    oracle's (IEEE division by absmax, then nearest codepoint)."""
    per_block = 63
    a = float(np.float32(absmax))
    end = start + count
    while start < end:
        n = min(per_block * chunk_blocks, end - start)
        nb = (n + per_block - 1) // per_block
        bits = torch.arange(start, start + nb * per_block, dtype=torch.int64, device="cuda")
        bits = torch.clamp(bits, max=end - 1)
        bits = torch.where(bits >= 1 << 31, bits - (1 << 32), bits)  # as signed 32-bit patterns
        vals = bits.to(torch.int32).view(torch.float32).view(nb, per_block)
        W = torch.cat([torch.full((nb, 1), a, device="cuda"), vals], dim=1).contiguous()
        q = capi.quantize_nf4(W.view(nb, 64), group=0)
        p = q.packed.view(nb, 32)
        idx = torch.stack([p >> 4, p & 15], dim=2).view(nb, 64)[:, 1:].reshape(-1)[:n]
        ref = oracle.nearest_codes_scaled_bits(start, n, a)
        got = idx.cpu().numpy()
        if not np.array_equal(got, ref):
            bad = int(np.flatnonzero(got != ref)[0])
            raise AssertionError(f"absmax {a!r}: weight bits {start + bad:#010x} -> "
                                 f"{got[bad]} (oracle {ref[bad]})")
        assert np.all(q.absmax_f32.cpu().numpy() == np.float32(a))
        start += n


def _sweep_all(absmax: float):
    """Every binary32 w with |w| <= absmax."""
    top = _f32_bits(absmax)
    _sweep(absmax, 0, top + 1)
    _sweep(absmax, 0x80000000, top + 1)


def _sweep_windows(absmax: float, half: int = 1 << 14):
    """Windows of 2 * half consecutive weights around w = th_k * absmax for
    every decision threshold th_k, plus the ends of the range."""
    a = float(np.float32(absmax))
    top = _f32_bits(a)
    for th in capi.nf4_thresholds():
        c = _f32_bits(float(np.float32(th) * np.float32(a)))
        mag, sign = c & 0x7FFFFFFF, c & 0x80000000
        lo, hi = max(0, mag - half), min(top, mag + half)
        _sweep(a, sign | lo, hi - lo + 1)
    for sign in (0, 0x80000000):
        _sweep(a, sign | max(0, top - half), min(top, half) + 1)
        _sweep(a, sign, min(top, half) + 1)


@pytest.mark.slow
@pytest.mark.parametrize("absmax", [1.0, 0.018737793, 1.5 * 2.0 ** -126, 1703.25, 9.1e-41],
                         ids=["1", "0.0187", "1.5e-126x2", "1703.25", "denormal"])
def test_exhaustive_decision_rule(absmax):
    """Every binary32 w in [-absmax, absmax] (about 2.1e9 values for absmax
    near 1) quantised as a non-maximal element of a block whose absmax is
    `absmax` gets the oracle's index: the division by the block constant
    and the nearest-codepoint rule, exactly."""
    _sweep_all(absmax)


@pytest.mark.parametrize("absmax", [2.0 ** -126, 2.0 ** -100, 0.5, 3.0517578e-05, 0.2718,
                                    2.0 ** 20, 6.02e23, 2.0 ** 126, 1.1e38, 3.4e38],
                         ids=lambda a: f"{a:.4g}")
def test_decision_rule_near_every_threshold(absmax):
    """Windows of 32768 consecutive weights around every decision threshold
    (scaled by the block constant), for powers of two, random constants and
    the ends of the binary32 range (where the reciprocal leaves the normal
    range and every element takes the IEEE quotient)."""
    _sweep_windows(absmax)
