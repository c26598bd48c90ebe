"""Reduced-precision input values, on the CPU: the rounding helpers against
torch's own conversions, and the accuracy bound of the variant.

The variant rounds each input value once to 16 bits (unit roundoff u: 2^-9
for bfloat16, 2^-11 for binary16) and then computes the exact cosine of the
rounded vectors.  A vector x + a with |a_k| <= u |x_k| is within angle
asin(u) of x, angles obey the triangle inequality and the cosine is
1-Lipschitz in the angle, so |cos(q', v') - cos(q, v)| <= 2 asin(u); the
float32 scores add at most the 2e-6 of the float32 path.
"""
import math

import numpy as np
import pytest

import oracle
from workload import CONFIGS, generate_rows
from workload.generate import CsrBatch
from workload.halfprec import (UNIT_ROUNDOFF, bf16_bits_to_f32, f16_bits_to_f32, to_bf16_bits,
                               to_f16_bits)

torch = pytest.importorskip("torch")


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100_000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100_000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, 1e-40], np.float32)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(to_bf16_bits(x), ref)
    back = bf16_bits_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_f16_rounding_matches_torch():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(100_000) * 10.0 ** rng.integers(-6, 4, 100_000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(to_f16_bits(x), ref)
    assert np.array_equal(f16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(torch.float16).float().numpy())


def _rounded(m, kind):
    bits = to_bf16_bits(m.values) if kind == "bf16" else to_f16_bits(m.values)
    vals = bf16_bits_to_f32(bits) if kind == "bf16" else f16_bits_to_f32(bits)
    return CsrBatch(m.indptr, m.indices, vals, m.dim)


@pytest.mark.parametrize("kind", ["bf16", "f16"])
def test_input_rounding_stays_within_the_bound(kind):
    cfg = CONFIGS["d65k_q1k_i10k"]
    Q, I = generate_rows(cfg, 0, 0, 200), generate_rows(cfg, 1, 0, 3000)
    exact = oracle.cosine(Q, I, f64=True)
    rounded = oracle.cosine(_rounded(Q, kind), _rounded(I, kind), f64=True)
    bound = 2 * math.asin(UNIT_ROUNDOFF[kind])
    err = float(np.abs(rounded - exact).max())
    assert err <= bound
    assert err > 0.0  # the rounding does change the scores
    # The post allows 16-bit data where an error below 1e-3 is acceptable
    # (section 5.3): binary16 meets it; bfloat16 does not on this workload,
    # which is why the bfloat16 variant is documented as outside that bar.
    if kind == "f16":
        assert err < 1e-3
    else:
        assert err > 1e-3


def test_binding_takes_16_bit_values_only_as_declared():
    sec = pytest.importorskip("sparse_embedding_exact_gb300")
    from sparse_embedding_exact_gb300 import _host_csr

    cfg = CONFIGS["d65k_q1k_i10k"]
    m = generate_rows(cfg, 0, 0, 20)
    _, keep = _host_csr(m)  # float32 by default
    assert keep[2].dtype == np.float32
    bits = to_bf16_bits(m.values)
    _, keep = _host_csr(CsrBatch(m.indptr, m.indices, bits, m.dim), "bf16")
    assert keep[2].dtype == np.uint16 and np.array_equal(keep[2], bits)  # passed through untouched
    h16 = m.values.astype(np.float16)
    _, keep = _host_csr(CsrBatch(m.indptr, m.indices, h16, m.dim), "f16")
    assert np.array_equal(keep[2], h16.view(np.uint16))
    for kind, vals in (("bf16", m.values), ("bf16", h16), ("f16", m.values)):
        with pytest.raises(TypeError):
            _host_csr(CsrBatch(m.indptr, m.indices, vals, m.dim), kind)
    assert sec._HOST_VALUES == {"f32": 0, "bf16": 1, "f16": 2}
