"""Arithmetic facts the GPU path relies on, checked on the CPU with exact
float64 arithmetic.

The Semantic-Unit Refresh scoring (Budgeted KV-Cache Repair for Evolving
Contexts, Sec. 7.3: fp32 scoring) runs on the bf16 tensor cores by writing the
normalised fp32 query as hi + mid + lo, three bf16 values: the split must be
exact, and a bf16 x bf16 product must be exact in fp32."""
import numpy as np

import oracle


def test_three_term_bf16_split_of_fp32_is_exact():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000).astype(np.float32) / np.float32(64)   # unit-norm query scale
    x = np.concatenate([x, np.float32([1.0, -1.0, 2.0 ** -20, -3.0e-8, 0.0])])
    hi = oracle.round_bf16(x.astype(np.float64))
    r1 = x.astype(np.float64) - hi
    assert np.all(r1.astype(np.float32).astype(np.float64) == r1)        # the remainder is an fp32 value
    mid = oracle.round_bf16(r1)
    lo_exact = r1 - mid
    lo = oracle.round_bf16(lo_exact)
    assert np.all(lo == lo_exact)                                         # the last term is a bf16 value
    assert np.all(hi + mid + lo == x.astype(np.float64))


def test_bf16_products_are_exact_in_fp32():
    rng = np.random.default_rng(1)
    a = oracle.round_bf16(rng.standard_normal(100000) * 3)
    b = oracle.round_bf16(rng.standard_normal(100000) / 7)
    p = a * b                                                             # exact in float64
    assert np.all(p.astype(np.float32).astype(np.float64) == p)
