"""The error bound behind the tolerance of the tensor-core importance passes.

fp32 operands reach the tensor cores as a bf16 high part hi = rn(x) and a
low part lo = rn(x - hi); a product keeps hi.hi + hi.lo + lo.hi.  The GPU
parity tests of the prefill importance producer rest on two facts checked
here on the host, in the same round-to-nearest-even conversion the packing
kernel uses:

* hi is within 2^-8 |x| of x, and the residual r = x - hi - lo of the split
  is at most 2^-17 |x| (x - hi is exact in fp32 and its leading bit lies at
  least 9 places below x's, so lo's 8 significant bits leave 2^-17);
* the three kept products differ from the exact product by at most
  2^-15 |q k| (dropped: lo.lo <= 2^-16, (hi + lo).r_k and r_q.k <= 2^-17
  each), so a D-term logit is off by at most 2^-15 * sum |q_d k_d| before
  accumulation, and typically by far less (the terms' errors have random
  signs; the median per-product error is near 2^-19).

Dropping any one of the three products breaks the bound by orders of
magnitude, so the check fails for a pass that forgets a term.
"""
import numpy as np
import torch

EPS_SPLIT = 2.0 ** -17


def split(x: np.ndarray):
    t = torch.from_numpy(x.astype(np.float32))
    hi = t.to(torch.bfloat16).to(torch.float32)
    lo = (t - hi).to(torch.bfloat16).to(torch.float32)
    return hi.numpy().astype(np.float64), lo.numpy().astype(np.float64)


def test_split_residual_within_2_pow_minus_17():
    rng = np.random.default_rng(0)
    mant = rng.uniform(-1.0, 1.0, 1 << 20)
    expo = rng.integers(-60, 60, mant.size)
    x = np.ldexp(mant, expo).astype(np.float32)
    x = np.concatenate([x, np.float32([1.0, -1.0, 0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9,
                                       np.nextafter(np.float32(1), np.float32(2))])])
    hi, lo = split(x)
    xd = x.astype(np.float64)
    # the high part alone is the bf16 rounding: half an ulp of 8 bits
    assert np.all(np.abs(xd - hi) <= 2.0 ** -8 * np.abs(xd))
    r = xd - hi - lo
    assert np.all(np.abs(r) <= EPS_SPLIT * np.abs(xd))
    # x - hi is exact in fp32, so the split is invariant under it
    assert np.all((x - hi.astype(np.float32)).astype(np.float64) == xd - hi)


def three_product_dot(q, k, keep=("hh", "hl", "lh")):
    qh, ql = split(q)
    kh, kl = split(k)
    terms = {"hh": qh * kh, "hl": qh * kl, "lh": ql * kh}
    return sum(terms[t] for t in keep).sum(axis=-1)


def test_three_products_within_2_pow_minus_15():
    rng = np.random.default_rng(1)
    for D in (64, 128):
        q = rng.uniform(-1.0, 1.0, (4096, D)).astype(np.float32)
        k = rng.uniform(-1.0, 1.0, (4096, D)).astype(np.float32)
        exact = (q.astype(np.float64) * k.astype(np.float64)).sum(axis=-1)
        mag = np.abs(q.astype(np.float64) * k.astype(np.float64)).sum(axis=-1)
        err = np.abs(three_product_dot(q, k) - exact)
        assert np.all(err <= 2.0 ** -15 * mag)
        # random signs: the typical logit error is far below the worst case
        assert np.median(err / mag) < 2.0 ** -19
    # one product at a time, over many pairs: the per-product bound holds
    # and is nearly reached
    x = rng.uniform(-1.0, 1.0, 1 << 20).astype(np.float32)
    y = rng.uniform(-1.0, 1.0, 1 << 20).astype(np.float32)
    exact = x.astype(np.float64) * y.astype(np.float64)
    rel = np.abs(three_product_dot(x[:, None], y[:, None]) - exact) / np.abs(exact)
    assert rel.max() <= 2.0 ** -15 and rel.max() > 2.0 ** -16


def test_dropping_a_product_breaks_the_bound():
    rng = np.random.default_rng(2)
    q = rng.uniform(-1.0, 1.0, (512, 128)).astype(np.float32)
    k = rng.uniform(-1.0, 1.0, (512, 128)).astype(np.float32)
    exact = (q.astype(np.float64) * k.astype(np.float64)).sum(axis=-1)
    mag = np.abs(q.astype(np.float64) * k.astype(np.float64)).sum(axis=-1)
    for keep in (("hh", "hl"), ("hh", "lh"), ("hh",)):
        err = np.abs(three_product_dot(q, k, keep) - exact)
        assert np.max(err / mag) > 8 * 2.0 ** -15, keep


def test_int8_operands_exact_in_bf16():
    """int8 caches take one product: every integer in [-128, 127] is exact
    in bf16 and a 128-term integer dot (< 2^21) is exact in fp32."""
    v = np.arange(-128, 128, dtype=np.float32)
    hi, lo = split(v)
    assert np.all(hi == v) and np.all(lo == 0)
    assert 128 * 128 * 128 < 2 ** 24
