"""Pins for the oracle's blockwise NF4 quantisation, double quantisation,
packing and dequantisation.

Pins used (none re-types the oracle's code):
  * closed forms printed on the pages: 4.5 bits/param without and ~4.127
    bits/param with double quantisation, ~3 GB saved at 65B ("QLoRA 的三个核心技术",
    double-quantisation paragraph); packed size (numel + 1) // 2
    ("QLoRA and 4bit Quantization | QLoRA 与 4-bit 量化", Step 4 ledger);
  * the page fixture of ch. 26 Step 4 (per-tensor scale 0.5, indices 0..11);
  * a hand-derived packing example (golden/pack_order_example.json);
  * exact rational arithmetic for the nearest codepoint of w / absmax;
  * library routines: numpy abs-max per block, torch's bf16 rounding;
  * invariants: the group maximum gets code 127, |a_hat - a| <= s2 / 2,
    round-trip error bound.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as orc


def _rand_w(rows, cols, seed, std=0.02):
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn(rows, cols, generator=g) * std).to(torch.bfloat16).float()
    return w.numpy()


def test_pack_order_hand_example(golden_dir):
    with open(os.path.join(golden_dir, "pack_order_example.json")) as f:
        ex = json.load(f)
    w = np.zeros((1, ex["block"]), dtype=np.float32)
    for k, v in ex["weights_nonzero"].items():
        w[0, int(k)] = v
    q = orc.quantize_nf4(w, block=ex["block"], group=0)
    assert list(q.idx[0, :4]) == ex["expected_indices_prefix"]
    assert [f"{b:02x}" for b in q.packed[:2]] == ex["expected_bytes_prefix_hex"]
    assert all(f"{b:02x}" == ex["expected_fill_byte_hex"] for b in q.packed[2:])
    assert q.absmax_f32[0] == np.float32(0.5)


def test_absmax_element_maps_to_endpoint():
    rng = np.random.default_rng(5)
    for sign, end in ((1.0, 15), (-1.0, 0)):
        w = rng.uniform(-0.01, 0.01, (2, 64)).astype(np.float32)
        w[1, 17] = sign * 0.05
        q = orc.quantize_nf4(w, group=0)
        assert q.idx[1, 17] == end
        assert q.absmax_f32[1] == np.float32(0.05)


def test_zero_block_maps_to_zero_codepoint():
    w = np.zeros((3, 128), dtype=np.float32)
    w[1, 70] = 0.3  # only block 3 (row 1, second half) is non-zero
    q = orc.quantize_nf4(w, group=256)
    zero_blocks = [0, 1, 2, 4, 5]
    idx = q.idx.reshape(-1, 64)
    for b in zero_blocks:
        assert np.all(idx[b] == 7)
        assert q.absmax_code[b] == 0
    assert q.absmax_code[3] == 127
    deq = orc.dequant_f32(q).reshape(-1, 64)
    for b in zero_blocks:
        assert np.all(deq[b] == 0.0)


def test_all_zero_matrix_gives_zero_scale():
    q = orc.quantize_nf4(np.zeros((4, 64), np.float32), group=256)
    assert q.scale2[0] == 0.0 and np.all(q.absmax_code == 0)
    assert np.all(q.packed == 0x77)


def test_block_absmax_matches_numpy():
    w = _rand_w(8, 256, 11)
    q = orc.quantize_nf4(w, group=0)
    expect = np.abs(w.reshape(-1, 64)).max(axis=1)
    assert np.array_equal(q.absmax_f32, expect)


def test_indices_are_exact_nearest_of_normalised_weight():
    """For each weight, w / a_block in exact arithmetic must be closest to the
    chosen codepoint, up to the binary32 rounding of the normalisation."""
    w = _rand_w(4, 128, 3)
    q = orc.quantize_nf4(w, group=0)
    cb = [Fraction(float(c)) for c in orc.codebook()]
    blocks = w.reshape(-1, 64)
    idx = q.idx.reshape(-1, 64)
    for b in range(blocks.shape[0]):
        a = Fraction(float(np.abs(blocks[b]).max()))
        for i in range(64):
            xn = Fraction(float(blocks[b, i])) / a
            d = [abs(xn - c) for c in cb]
            m = min(d)
            slack = Fraction(2) ** -22
            ok = {k for k, dk in enumerate(d) if dk - m <= slack}
            assert idx[b, i] in ok


def test_dq_group_max_has_code_127_and_error_bound():
    w = _rand_w(64, 512, 7)  # 512 blocks -> 2 groups of 256
    q = orc.quantize_nf4(w, group=256)
    a = np.abs(w.reshape(-1, 64)).max(axis=1)
    for g in range(2):
        ag = a[g * 256:(g + 1) * 256]
        codes = q.absmax_code[g * 256:(g + 1) * 256]
        s2 = q.scale2[g]
        assert codes[np.argmax(ag)] == 127
        assert np.all(codes >= 0)
        ahat = codes.astype(np.float64) * np.float64(s2)
        assert np.all(np.abs(ahat - ag) <= s2 / 2 * (1 + 1e-6))
        # s2 is the group max over 127 to within binary32 rounding
        assert abs(float(s2) - float(ag.max()) / 127) <= 2 ** -23 * float(s2)


def test_partial_last_group():
    w = _rand_w(5, 64 * 60, 9)  # 300 blocks -> groups of 256 and 44
    q = orc.quantize_nf4(w, group=256)
    assert q.scale2.size == 2
    a = np.abs(w.reshape(-1, 64)).max(axis=1)
    assert q.absmax_code[256 + np.argmax(a[256:])] == 127


def test_storage_closed_forms(golden_dir):
    with open(os.path.join(golden_dir, "storage_closed_forms.json")) as f:
        ex = json.load(f)
    for rows, cols in ((4096, 4096), (14336, 4096), (4096, 14336), (256, 256 * 64)):
        p, c, s = orc.storage_bytes(rows, cols, 64, 256)
        n = rows * cols
        bits_dq = 8 * (p + c + s) / n
        assert bits_dq == 4.126953125  # 4 + 8/64 + 32/(64*256)
        assert round(bits_dq, ex["printed_decimals_dq"]) == ex["bits_per_param_dq_printed"]
        p0, c0, s0 = orc.storage_bytes(rows, cols, 64, 0)
        assert 8 * (p0 + c0 + s0) / n == ex["bits_per_param_no_dq_printed"]
    # 65B model: saving of double quantisation, printed as about 3 GB
    n65 = ex["params_65b"]
    saving_gb = n65 * (4.5 - 4.126953125) / 8 / 1e9
    assert abs(saving_gb - ex["saving_65b_gb_printed"]) / ex["saving_65b_gb_printed"] <= \
        ex["saving_65b_gb_rel_tol"]
    # packed bytes rule from the page ledger, odd element count included
    for n in (1, 2, 7, 12, 4096):
        assert orc.storage_bytes(1, n, 1, 0)[0] == (n + 1) // 2


def test_quantize_buffer_sizes_match_closed_form():
    w = _rand_w(16, 1024, 1)
    q = orc.quantize_nf4(w, group=256)
    p, c, s = orc.storage_bytes(16, 1024, 64, 256)
    assert q.packed.nbytes == p and q.absmax_code.nbytes == c and q.scale2.nbytes == s


def test_p1_fixture_dequant(golden_dir):
    """Page fixture: indices 0..11 in a 3x4 matrix, per-tensor scale 0.5.
    The per-tensor scale is expressed as one binary32 constant per 4-wide
    block (no double quantisation)."""
    with open(os.path.join(golden_dir, "p1_fixture.json")) as f:
        fx = json.load(f)
    idx = np.array(fx["indices"], dtype=np.uint8)
    rows, cols = idx.shape
    packed = ((idx.reshape(-1)[0::2] << 4) | idx.reshape(-1)[1::2]).astype(np.uint8)
    q = orc.NF4Weight(rows, cols, cols, 0, packed, np.zeros(0, np.int8),
                      np.full(rows, fx["scale"], np.float32), np.zeros(0, np.float32),
                      idx, 0)
    got = orc.dequant_bf16(q)
    table = torch.tensor(orc.codebook())
    ref = (table[torch.tensor(idx).long()] * fx["scale"]).to(torch.bfloat16)
    assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))
    assert got.shape == idx.shape
    assert np.all(np.isfinite(orc.bf16_bits_to_f32(got)))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    vals = [rng.normal(0, 1, 20000).astype(np.float32),
            rng.normal(0, 1e-30, 1000).astype(np.float32),
            np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                      1e-45, -1e-45, 1.0, -1.0], np.float32)]
    # exact ties: low 16 bits == 0x8000 with both parities of bit 16
    hi = rng.integers(0, 0x7f00, 2000, dtype=np.uint32) << 16
    vals.append((hi | 0x8000).view(np.float32))
    vals.append((hi | 0x18000).view(np.float32))
    v = np.concatenate(vals)
    got = orc.bf16_rne(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_dequant_roundtrip_error_bound():
    """|w_hat - w| <= a * (max half gap of the codebook) + s2/2 + bf16 rounding."""
    w = _rand_w(32, 512, 21)
    q = orc.quantize_nf4(w, group=256)
    deq = orc.dequant_f32(q).astype(np.float64)
    cb = orc.codebook().astype(np.float64)
    half_gap = np.max(np.diff(cb)) / 2
    a = np.abs(w.reshape(-1, 64)).max(axis=1).repeat(64).reshape(w.shape)
    s2 = np.repeat(q.scale2, 256 * 64)[: w.size].reshape(w.shape)
    bound = a * half_gap + s2 / 2 + np.abs(deq) * 2 ** -8 + 1e-12
    assert np.all(np.abs(deq - w) <= bound)
    # and the error is far below the scale of the weights on average
    assert np.sqrt(np.mean((deq - w) ** 2)) < 0.2 * np.std(w)


def test_dequant_uses_group_scale_of_each_block():
    """Two groups with very different magnitudes: every dequantised block
    must land in its own group's range (catches a wrong group index)."""
    w = np.concatenate([_rand_w(4, 64 * 64, 2, std=0.001), _rand_w(4, 64 * 64, 3, std=1.0)])
    q = orc.quantize_nf4(w, group=256)
    deq = orc.dequant_f32(q)
    assert np.abs(deq[:4]).max() < 0.01 and np.abs(deq[4:]).max() > 1.0
    assert np.abs(deq - w).max() <= 0.16 * np.abs(w).max()


def test_nonfinite_inputs_are_counted():
    w = _rand_w(2, 64, 4)
    w[1, 3] = np.inf
    w[0, 0] = np.nan
    q = orc.quantize_nf4(w, group=0)
    assert q.nonfinite == 2


def test_quantize_rejects_bad_shapes():
    with pytest.raises(ValueError):
        orc.quantize_nf4(np.zeros((2, 65), np.float32))
    with pytest.raises(ValueError):
        orc.quantize_nf4(np.zeros((2, 64), np.float32), block=63)


# ------------------------------------------------------------- block 128
# "QLoRA and 4bit Quantization | QLoRA 与 4-bit NormalFloat 量化核心机制",
# engineering notes: 64 or 128 parameters share one scale.

def test_block128_storage_closed_forms():
    """128-weight blocks: 4 + 32/128 = 4.25 bits per parameter with binary32
    constants, 4 + 8/128 + 32/(128*256) with double quantisation."""
    for rows, cols in ((4096, 4096), (14336, 4096), (4096, 14336)):
        n = rows * cols
        p0, c0, s0 = orc.storage_bytes(rows, cols, 128, 0)
        assert 8 * (p0 + c0 + s0) / n == 4.25
        p, c, s = orc.storage_bytes(rows, cols, 128, 256)
        assert 8 * (p + c + s) / n == 4 + 8 / 128 + 32 / (128 * 256)


def test_block128_absmax_and_brute_force_nearest():
    """Per 128-weight block the constant is numpy's abs-max over the block,
    and every index is the nearest codepoint of w / a found by brute force
    over the 16 entries (exact rationals, up to the binary32 rounding of the
    division)."""
    w = _rand_w(3, 256, 21)
    w[1, 128 + 5] = 0.0
    w[2, :128] = 0.0  # an all-zero block
    q = orc.quantize_nf4(w, block=128, group=0)
    blocks = w.reshape(-1, 128)
    assert np.array_equal(q.absmax_f32, np.abs(blocks).max(axis=1))
    cb = [Fraction(float(c)) for c in orc.codebook()]
    idx = q.idx.reshape(-1, 128)
    for b in range(blocks.shape[0]):
        a = Fraction(float(np.abs(blocks[b]).max()))
        for i in range(128):
            if a == 0:
                assert idx[b, i] == 7
                continue
            xn = Fraction(float(blocks[b, i])) / a
            d = [abs(xn - c) for c in cb]
            m = min(d)
            ok = {k for k, dk in enumerate(d) if dk - m <= Fraction(2) ** -22}
            assert idx[b, i] in ok
    # one block of 128 is not two blocks of 64: the halves share one constant
    w2 = np.zeros((1, 128), np.float32)
    w2[0, 0], w2[0, 100] = 0.02, 0.2
    q128 = orc.quantize_nf4(w2, block=128, group=0)
    q64 = orc.quantize_nf4(w2, block=64, group=0)
    assert q128.absmax_f32.tolist() == [np.float32(0.2)]
    assert q128.idx[0, 0] != q64.idx[0, 0]
