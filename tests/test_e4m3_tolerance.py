"""The E4M3 code comparison used by the GPU read-copy tests, checked on the
CPU: codes decided in fp32 (a factor 448 / amax and a product, each rounded,
the kernels' arithmetic) pass against the oracle's double-precision codes,
and planted errors (two steps, a flipped sign, one step away from any tie)
are rejected."""
import pytest
import torch

import oracle
from ssu_testlib import assert_e4m3_codes_close


def _fp32_codes(st: torch.Tensor) -> torch.Tensor:
    amax = st.abs().amax(dim=-1, keepdim=True)
    factor = torch.where(amax > 0, 448.0 / torch.where(amax > 0, amax, torch.ones_like(amax)),
                         torch.ones_like(amax))
    return (st * factor).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.fixture(scope="module")
def pool():
    g = torch.Generator().manual_seed(5)
    return torch.randn((64, 4, 16, 128), generator=g) * torch.rand((64, 4, 16, 1), generator=g) * 3


def test_fp32_decided_codes_pass(pool):
    want, _ = oracle.shadow_refresh(pool, oracle.SHADOW_E4M3)
    got = _fp32_codes(pool)
    assert (got != want).sum() < 0.001 * got.numel()
    assert_e4m3_codes_close(got, want, pool)


@pytest.mark.parametrize("planted", ["two_steps", "sign", "off_tie"])
def test_planted_code_errors_fail(pool, planted):
    want, _ = oracle.shadow_refresh(pool, oracle.SHADOW_E4M3)
    got = want.clone()
    i = (3, 2, 5, 17)
    c = int(got[i])
    if planted == "two_steps":
        got[i] = (c & 0x80) | min((c & 0x7F) + 2, 0x7E)
    elif planted == "sign":
        got[i] = c ^ 0x80 if c & 0x7F else 0x81
    else:
        got[i] = (c & 0x80) | ((c & 0x7F) + 1 if (c & 0x7F) < 0x7E else (c & 0x7F) - 1)
    with pytest.raises(AssertionError):
        assert_e4m3_codes_close(got, want, pool)
