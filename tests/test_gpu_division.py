"""The quantizer divides by its float16 scale through a correctly rounded reciprocal and one
exact-remainder correction (Markstein's theorem) instead of an IEEE division; the library's
own device self-check compares the two on every finite bf16 dividend with every positive
finite float16 scale, plus 2^29 hashed float32 dividends, and must find no difference."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_scale_division_equals_ieee_division():
    import bit_rotated_kv_gb300 as kvq
    bad = torch.zeros(1, dtype=torch.int64, device="cuda")
    kvq.kvq_selftest_scale_division(bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
