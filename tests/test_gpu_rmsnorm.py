"""gdn_rmsnorm (the layer's input RMSNorm, optionally fused with the residual add) against the fp64
oracle: the residual stream bit for bit, U element by element, over ragged hidden sizes up to the
largest supported (8192), the layer's 5120 at decode and prefill-like token counts, in place."""
import numpy as np
import pytest
import torch

from oracle import oracle
from tests import gdnutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


def _case(T, Dh, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = U.synth.bf16_bits((scale * rng.normal(size=(T, Dh))).astype(np.float32))
    r = U.synth.bf16_bits((4.0 * rng.normal(size=(T, Dh))).astype(np.float32))
    g = rng.uniform(0.5, 1.5, size=Dh).astype(np.float32)
    return x, r, g


@pytest.mark.parametrize("T,Dh,with_res", [(1, 8, False), (37, 1000, True), (256, 5120, True),
                                           (3, 8192, True), (1031, 5120, False)])
def test_rmsnorm_matches_oracle(b, T, Dh, with_res):
    x, r, g = _case(T, Dh, 100 + T)
    out = torch.zeros((T, Dh), dtype=torch.bfloat16, device="cuda")
    res = U.dev_bf16(r) if with_res else None
    b.gdn_rmsnorm(U.dev_bf16(x), U.dev(g), 1e-6, out, residual=res)
    u_ref, res_ref = oracle.rmsnorm(x, g, 1e-6, r if with_res else None)
    U.check_out(U.host_f64_from_bf16(out), u_ref, "U")
    if with_res:
        np.testing.assert_array_equal(U.host_bits(res), res_ref)


def test_rmsnorm_in_place_and_tiny_rows(b):
    """out = x (in place) with the residual; rows whose values are tiny, so eps dominates."""
    T, Dh = 64, 5120
    x, r, g = _case(T, Dh, 140)
    x[::7] = U.synth.bf16_bits(np.full((1, Dh), 1e-5, np.float32))  # mean square 1e-10 << eps
    xd, rd = U.dev_bf16(x), U.dev_bf16(r)
    b.gdn_rmsnorm(xd, U.dev(g), 1e-6, xd, residual=rd)
    u_ref, res_ref = oracle.rmsnorm(x, g, 1e-6, r)
    U.check_out(U.host_f64_from_bf16(xd), u_ref, "U in place")
    np.testing.assert_array_equal(U.host_bits(rd), res_ref)
    u_ref2, _ = oracle.rmsnorm(x[::7], g, 1e-6)
    x2 = U.dev_bf16(x[::7].copy())
    out2 = torch.zeros_like(x2)
    b.gdn_rmsnorm(x2, U.dev(g), 1e-6, out2)
    U.check_out(U.host_f64_from_bf16(out2), u_ref2, "eps-dominated rows")


def test_rmsnorm_no_tokens(b):
    g = torch.ones(5120, dtype=torch.float32, device="cuda")
    empty = torch.zeros((0, 5120), dtype=torch.bfloat16, device="cuda")
    b.gdn_rmsnorm(empty, g, 1e-6, empty)
