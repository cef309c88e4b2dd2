"""Failure detection without a GPU fault: a wait that nothing completes runs
out its bounded limit, the kernel records a device timeout in the error
word and returns, the host reads RLK_ERR_DEVICE_TIMEOUT, the word is
cleared, and the same context then runs the hot path correctly."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import lib, torch_cuda

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    torch = torch_cuda()
    rlk = lib()
    rlk.rlk_attn_check_device_error()  # a clean error word to start from
    rlk.rlk_attn_selftest_wait_timeout()
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_check_device_error()
    assert e.value.status == 6  # RLK_ERR_DEVICE_TIMEOUT
    assert "0x7e1" in rlk.rlk_attn_last_error()
    rlk.rlk_attn_check_device_error()  # reading the word cleared it
    # the context is intact: a RoPE pass still matches the oracle bit for bit
    from deterministic_context_attention_gb300 import device as dv
    cu = synth.cu_seqlens([100, 37])
    x = synth.normal_bf16(61, synth.T_Q, (137, 8, 128))
    xd = dv.bf16_to_device(x)
    table = torch.from_numpy(rlk.rlk_attn_rope_table(1.0e6, 100)).cuda()
    rlk.rlk_attn_rope(rlk.make_params(2), xd, xd, 8, cu, None, table, 100)
    rlk.rlk_attn_check_device_error()
    pos = np.concatenate([np.arange(100), np.arange(37)]).astype(np.int32)
    np.testing.assert_array_equal(xd.float().cpu().numpy(), oracle.rope_f32(x, pos, 1.0e6))
