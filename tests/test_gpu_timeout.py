"""The failure path of the bounded device waits, without a GPU fault: a wait on
an mbarrier phase that nothing completes gives up after its limit, the device
error word reports ATTN_ETIMEOUT to the host, and the context stays usable."""
import pytest
import torch

from block_sparse_attention_online_gb300 import binding as bs
from block_sparse_attention_online_gb300 import workloads as W
from tests.test_gpu_decode import check_decode

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    bs.attn_skip_last_device_error()  # start from a clear error word
    bs.attn_skip_selftest_wait_timeout()
    with pytest.raises(bs.AttnSkipError) as e:
        bs.attn_skip_last_device_error()
    assert e.value.status == bs.ATTN_ETIMEOUT
    bs.attn_skip_last_device_error()  # the word was cleared by the read
    # the context still runs the real kernels correctly
    cfg = W.GQA_DECODE_32K.with_(B=2, L=1500, n_splits=3, seed=91)
    q, k, v = W.decode_inputs(cfg)
    check_decode(cfg, q, k, v, 1e-9)
    torch.cuda.synchronize()
