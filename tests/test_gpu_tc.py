"""GPU parity of the tensor-core (tcgen05) grouped expert GEMM (-m gpu).

Experts that receive more than 32 tokens are computed by the tcgen05 kernel
in units of <= 128 tokens; these cases route enough tokens to each expert
to take that path, from the smallest one (one super-block of K, one 128-row
tile, 33 tokens) upwards, and compare the whole layer with the CPU oracle.
"""
import pytest

from test_gpu_moe import MOE_TOL, NVFP4, Q4_K, Q6_K, Q8_0, _moe_case, dq  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,E,k,H,F,ns,T,xdt", [
    (Q4_K, 1, 1, 256, 256, 0, 33, 1),       # one unit of 33 tokens: N = 48, 2 boxes
    (Q4_K, 1, 1, 512, 512, 1, 40, 2),       # shared expert too; 4 row tiles
    (Q8_0, 1, 1, 256, 256, 0, 130, 1),      # > 128 tokens: two units (128 + 2)
    (Q6_K, 1, 1, 2048, 2048, 0, 64, 2),     # Q6_K rows, bf16 activations
    (NVFP4, 1, 1, 512, 256, 1, 150, 2),     # NVFP4 rows: two units, shared expert
])
def test_tc_wide_units(dq, orc, fmt, E, k, H, F, ns, T, xdt):
    err, _ = _moe_case(dq, orc, fmt, E, k, H, F, ns, T, xdt, seed=7000 + T + E)
    assert err <= MOE_TOL, err
