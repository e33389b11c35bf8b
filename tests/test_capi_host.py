"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, and its host-side tables agree with what the pages fix and with the
oracle's decision rule.  No GPU needed (no compute call is made)."""
import ctypes
import os
import re
import struct

import numpy as np
import pytest

from bit_nf4_quantized_35_b300 import build as libbuild
from bit_nf4_quantized_35_b300 import capi
from oracle import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return capi.load()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "qlora.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qlora_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = header_symbols()
    for name in ("qlora_quantize_nf4", "qlora_dequant", "qlora_linear_fwd", "qlora_linear_bwd"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in header_symbols() if not hasattr(lib, s)]
    assert not missing, missing
    assert set(header_symbols()) == set(capi.EXPORTED)


def test_codebook_matches_printed_table(lib, golden_dir):
    cb = np.array(capi.nf4_codebook(), dtype=np.float32)
    ref = oracle.codebook()
    assert cb.tobytes() == ref.tobytes()
    assert cb[7] == 0.0 and cb[0] == -1.0 and cb[15] == 1.0


def _f32_from_bits(b):
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def _bits(f):
    return struct.unpack("<I", struct.pack("<f", f))[0]


def test_thresholds_reproduce_oracle_rule_near_every_boundary(lib):
    """index = #thresholds <= x must equal the oracle's first-argmin of fp32
    distances for every fp32 within 2^12 ulps of each threshold."""
    th = np.array(capi.nf4_thresholds(), dtype=np.float32)
    assert np.all(np.diff(th) > 0)
    cb = oracle.codebook()
    for k in range(15):
        assert cb[k] < th[k] <= cb[k + 1]
        start = _bits(float(th[k])) - 4096
        bits = np.arange(start, start + 8193, dtype=np.int64).astype(np.uint32)
        xs = bits.view(np.float32)
        xs = xs[np.isfinite(xs) & (np.abs(xs) <= 1)]
        ours = np.searchsorted(th, xs, side="right")
        ref = np.array([oracle.nearest_code(float(x)) for x in xs[::64]])
        assert np.array_equal(ours[::64], ref)
        # dense check through the oracle's bit-range routine
        lo = int(bits.min())
        ref_dense = oracle.nearest_codes_bits(lo, 8193)
        xs_dense = np.arange(lo, lo + 8193, dtype=np.int64).astype(np.uint32).view(np.float32)
        ours_dense = np.searchsorted(th, xs_dense, side="right")
        assert np.array_equal(ours_dense, ref_dense), k


def test_thresholds_random_sample(lib):
    th = np.array(capi.nf4_thresholds(), dtype=np.float32)
    rng = np.random.default_rng(7)
    xs = rng.uniform(-1, 1, 200_000).astype(np.float32)
    ours = np.searchsorted(th, xs, side="right")
    ref = np.array([oracle.nearest_code(float(x)) for x in xs[:5000]])
    assert np.array_equal(ours[:5000], ref)


def test_worked_example_through_thresholds(lib, golden_dir):
    import json
    ex = json.load(open(os.path.join(golden_dir, "worked_example.json")))
    th = np.array(capi.nf4_thresholds(), dtype=np.float32)
    idx = int(np.searchsorted(th, np.float32(ex["normalised_value"]), side="right"))
    assert idx == ex["index_in_printed_table"]


@pytest.mark.parametrize("rows,cols,group", [(4096, 4096, 256), (14336, 4096, 256),
                                             (256, 256, 0), (3, 128, 64)])
def test_sizes_match_oracle_storage(lib, rows, cols, group):
    assert capi.nf4_sizes(rows, cols, 64, group) == oracle.storage_bytes(rows, cols, 64, group)


def test_sizes_reject_bad_shapes(lib):
    with pytest.raises(capi.QloraError):
        capi.nf4_sizes(4, 100, 64, 256)


def test_workspace_size_monotone(lib):
    a = capi.workspace_size(16, 4096, 4096, 16)
    b = capi.workspace_size(8192, 4096, 4096, 16)
    assert 0 < a < b


def test_quantile_codebook_matches_oracle(lib):
    """The library's quantile-formula table (Wichura AS 241 on the host)
    equals the oracle's (bisection on the normal CDF) bit for bit."""
    cb = np.array(capi.nf4_codebook(capi.QLORA_CODEBOOK_QUANTILE), dtype=np.float32)
    assert cb.tobytes() == oracle.codebook(1).tobytes()


def test_quantile_thresholds_reproduce_oracle_rule(lib):
    th = np.array(capi.nf4_thresholds(capi.QLORA_CODEBOOK_QUANTILE), dtype=np.float32)
    cb = oracle.codebook(1)
    assert np.all(np.diff(th) > 0)
    for k in range(15):
        assert cb[k] < th[k] <= cb[k + 1]
        start = _bits(float(th[k])) - 512 if th[k] > 0 else _bits(float(th[k])) - 512
        bits = np.arange(start, start + 1025, dtype=np.int64).astype(np.uint32)
        xs = bits.view(np.float32)
        xs = xs[np.isfinite(xs) & (np.abs(xs) <= 1)]
        ours = np.searchsorted(th, xs, side="right")
        ref = np.array([oracle.nearest_code_cb(1, float(x)) for x in xs])
        assert np.array_equal(ours, ref), k
    rng = np.random.default_rng(8)
    xs = rng.uniform(-1, 1, 20000).astype(np.float32)
    ref = np.array([oracle.nearest_code_cb(1, float(x)) for x in xs])
    assert np.array_equal(np.searchsorted(th, xs, side="right"), ref)


def test_unknown_codebook_is_rejected(lib):
    with pytest.raises(capi.QloraError):
        capi.nf4_codebook(2)
