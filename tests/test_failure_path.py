"""GPU test of the failure path, made without any GPU fault: a test hook
withholds one TMA load of the next attention launch and shortens every wait
of that launch to 20 ms.  The launch must give up, report device error 2
through the host-readable error word, leave the context usable, and the next
launch must run clean and match the oracle."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from helpers import assert_bf16_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def T():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_attention_iha_gb300 as T
    T.lib()
    return T


def test_withheld_load_times_out_and_next_launch_is_clean(T):
    import torch
    q, k, v = (S.normal((1, 600, 4, 128), 41, c) for c in range(3))
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    assert T.device_error(clear=True) == 0
    assert T.lib().iha_test_fail_next_wait(20000) == 0      # 20 ms limit, one launch
    out = torch.zeros((1, 600, 4, 128), dtype=torch.bfloat16, device="cuda")
    T.mha_fwd(qd, kd, vd, mask=T.MASK_CAUSAL, out=out)
    assert T.device_error(clear=True) == 2                   # a bounded wait gave up
    assert T.device_error() == 0                             # and the word clears
    # the hook was one-shot: the next launch runs normally and is correct
    o = T.mha_fwd(qd, kd, vd, mask=T.MASK_CAUSAL)
    torch.cuda.synchronize()
    assert T.device_error() == 0
    ro, _ = O.attention(q[:, None], k[:, None], v[:, None], O.MASK_CAUSAL)
    assert_bf16_close(to_f64(o), ro[:, 0], "after the failed launch")


def test_hook_rejects_out_of_range_limit(T):
    assert T.lib().iha_test_fail_next_wait(0) == 1
    assert T.lib().iha_test_fail_next_wait(2_000_000) == 1
