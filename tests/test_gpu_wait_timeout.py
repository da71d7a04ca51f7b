"""The bounded-wait error path, exercised without any fault (no trap, no bad
address, no endless loop): a test hook makes the CTA-pair decode kernel's
producers stop issuing weight stages part-way and shortens every wait bound
to 20 ms. The copies already issued land; the consumers waiting for the
stages never issued give up, record WQ_ETIMEOUT and finish the kernel. The
host reads the status, the context stays usable, and the next normal call is
correct."""

import numpy as np
import pytest

import oracle as O
import wq_inputs as I
from helpers import assert_bf16_close, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int2_gb300 as wq  # noqa: E402


@pytest.mark.parametrize("stop_stage", [0, 3, 19])
def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_is_correct(stop_stage):
    lib = wq.load()
    M, N, K, bits = 1, 17408, 5120, 6
    assert wq.debug_route(M, N, K, bits, torch.cuda.get_device_properties(0).multi_processor_count) == \
        "decode_pair"
    x = I.make_x(M, K, 600)
    q = I.make_codes(N, K, bits, 601)
    s = I.make_scales(N, K // 128, 602)
    packed, s_dev = wq.wna16_repack(to_dev(q), to_dev_bf16(s), bits)
    xd = to_dev_bf16(x)
    wq.check_status()                                     # clean start
    assert lib.wq_debug_decode_wait_fault(stop_stage, 20_000_000) == 0
    try:
        wq.wna16_gemm(xd, packed, s_dev, N, K, bits)       # enqueues fine; its waits will run out
        with pytest.raises(wq.WQError) as err:
            wq.check_status()
        assert err.value.status == 4                       # WQ_ETIMEOUT
    finally:
        assert lib.wq_debug_decode_wait_fault(-1, 0) == 0
    wq.check_status()                                     # the status word was cleared
    ns = np.random.default_rng(stop_stage).choice(N, 64, replace=False)
    y = wq.wna16_gemm(xd, packed, s_dev, N, K, bits)
    torch.cuda.synchronize()
    got = y[:, torch.as_tensor(ns, device="cuda")]
    assert_bf16_close(got, O.wna16_ref(x, q[ns], s[ns], bits), "after the timeout")
    wq.check_status()
